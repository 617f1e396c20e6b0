/*
 * tk.h -- C ABI of libtk: byte-level BPE encoding on one GB300 (sm_103a).
 *
 * The library encodes typed text segments into token ids with a tiktoken-style
 * encoding: a bytes->rank table whose rank is the id, the cl100k split pattern,
 * and a dict of special tokens ("tiktoken Deep Dive", "An encoding is three
 * objects, not a model").  One call encodes a whole prompt of ordered
 * (text, allow_special) segments ("Making Kimi K3 Tokenization 18x Faster For
 * Million Token Agentic Workloads", "One native call for the whole serving
 * path"); every step of the encode runs in CUDA kernels, ordered on the
 * caller's stream.
 *
 * Conventions
 *   - "d_" pointers are device pointers, "h_" pointers are host pointers.
 *   - The caller owns every input and output buffer.  tk_load copies its
 *     tables into library-owned device memory; a workspace owns the scratch
 *     of one encode in flight (one workspace per concurrent stream).
 *   - Every function returns TK_OK (0) or a negative TK_E_* code, and leaves
 *     outputs unspecified on error.  tk_last_error() gives a one-line message
 *     for the calling thread's last failure.
 *   - Ids are int32; token byte offsets are int64.  Texts are limited to
 *     2^31 - 1024 bytes per call.
 */
#ifndef TK_H
#define TK_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct tk_tokenizer tk_tokenizer;
typedef struct tk_workspace tk_workspace;

enum {
  TK_OK = 0,
  TK_E_ARG = -1,      /* bad argument (null pointer, negative size, unknown pattern) */
  TK_E_TABLE = -2,    /* rank/special table rejected by tk_load */
  TK_E_UTF8 = -3,     /* input text is not valid UTF-8 (position in tk_last_error) */
  TK_E_CAPACITY = -4, /* output buffer too small; the required size is still returned */
  TK_E_CUDA = -5,     /* a CUDA runtime call failed */
  TK_E_NOMEM = -6,    /* host or device allocation failed */
  TK_E_TIMEOUT = -7,  /* a bounded device-side wait gave up (never expected) */
  TK_E_BADID = -8,    /* tk_decode met an id that is neither a rank nor a special */
  TK_E_LIMIT = -9     /* input exceeds the workspace's max_bytes / max_segments */
};

enum { TK_PATTERN_CL100K = 1, TK_PATTERN_R50K_DIGITS = 2 };

/*
 * tk_load -- build a tokenizer from host arrays (copied; the caller may free
 * them on return).
 *
 *   rank_bytes, rank_off[n+1], rank_ids[n]: mergeable token i is
 *       rank_bytes[rank_off[i] .. rank_off[i+1]) with rank (= id) rank_ids[i]
 *       ("tiktoken Deep Dive", "An encoding is three objects": one map
 *       bytes -> rank where the rank is the token id).  rank_off[0] must be 0.
 *   spec_bytes, spec_off[n_spec+1], spec_ids[n_spec]: special tokens, matched
 *       by exact string outside the merge loop ("Special tokens and the
 *       injection nobody plans for").  May be empty (n_spec = 0).
 *   pattern_id: TK_PATTERN_CL100K, the pattern printed in "tiktoken Deep
 *       Dive", "The split pattern"; or TK_PATTERN_R50K_DIGITS, the same
 *       alternation with r50k's digit clause " ?\p{N}++" (an unbounded digit
 *       run with an optional leading space; "r50k, cl100k, o200k") in place
 *       of cl100k's \p{N}{1,3}+.
 *
 * Rejected with TK_E_TABLE: a missing single byte ("The byte floor": all 256
 * bytes must be tokens), duplicate token bytes, duplicate ids, ids >= 2^20 - 1,
 * empty tokens, specials longer than 64 bytes or not valid UTF-8, special ids
 * that collide with ranks, and specials that can overlap one another in text
 * (a suffix of one equal to a prefix of another, or one inside another).
 * The handle is immutable after load and may be shared across threads.
 */
int tk_load(const uint8_t* rank_bytes, const int64_t* rank_off, const uint32_t* rank_ids,
            int64_t n, const uint8_t* spec_bytes, const int64_t* spec_off,
            const int32_t* spec_ids, int64_t n_spec, int pattern_id, tk_tokenizer** out);

void tk_free(tk_tokenizer* tok);

/*
 * tk_workspace_create -- allocate the device scratch for encodes of up to
 * max_bytes bytes in up to max_segments segments ("tokenizers v1: encode,
 * decode and scaling, measured", "Key Technical Improvements": the merge
 * working set lives in a caller-owned scratch buffer, so an encode never
 * touches an allocator).  About 44 bytes of device memory per byte of
 * max_bytes (11.9 GB for max_bytes = 256 MiB: seven 4-byte arrays indexed
 * by byte position for the long-piece merges, the per-tile staging of the
 * ids, the host-call staging, the mid-piece lists and the bitmaps).  A
 * workspace serves one encode at a time.
 */
int tk_workspace_create(const tk_tokenizer* tok, int64_t max_bytes, int64_t max_segments,
                        tk_workspace** out);

void tk_workspace_free(tk_workspace* ws);

/*
 * tk_encode_segments -- encode S ordered segments in one call.
 *
 *   d_text[n_bytes]: the segments' UTF-8 bytes, concatenated.
 *   d_seg_off[S+1]: segment s is d_text[d_seg_off[s] .. d_seg_off[s+1]);
 *       d_seg_off[0] = 0, non-decreasing, d_seg_off[S] = n_bytes.
 *   d_allow_special[S]: 1 = special strings in this segment become their
 *       special ids; 0 = they are ordinary text ("Making Kimi K3
 *       Tokenization ...", "Why Kimi K3 tokenization is non-trivial": user and
 *       tool text keeps literal control strings as text).
 *   tiktoken_safe: 1 = first cut each segment into windows of at most 400,000
 *       characters, then cut runs of white-space or non-white-space
 *       characters at 25,000 characters ("One native call for the whole
 *       serving path"); each piece is encoded on its own.
 *   d_out_ids[out_capacity]: receives the ids in input order.
 *       out_capacity >= n_bytes always suffices (every token covers >= 1 byte).
 *   d_out_offsets[S+1]: segment s's ids are d_out_ids[d_out_offsets[s] ..
 *       d_out_offsets[s+1]); d_out_offsets[S] is the total.
 *   h_n_ids: receives the total number of ids (also when it exceeds
 *       out_capacity, in which case TK_E_CAPACITY is returned).
 *   cuda_stream: a cudaStream_t (NULL = legacy default stream).  The encode
 *       is ordered on this stream: the kernels of the pre-tokens of 5 bytes
 *       or more run on the workspace's side streams, forked from and joined
 *       back into cuda_stream by events, so work queued on cuda_stream before
 *       the call is seen and work queued after it waits for the whole encode.
 *       The one device->host status read goes on cuda_stream (on the graph's
 *       stream for a replayed call, below); the call returns after that read
 *       completes.
 *
 * Repeated calls: when a workspace sees the same arguments (tokenizer,
 * buffer addresses, sizes, tiktoken_safe, attached cache) a second time in a
 * row, for a call under 16 MiB, it captures the call's launches into a CUDA
 * graph and replays it from then on (on a stream of its own, joined with cuda_stream by events, with
 * the same ordering as above).  The buffers' contents may change between
 * calls; the graph reads them when it runs.  Calls with per-kernel profiling
 * on, and every call after a capture that failed, launch directly.
 *
 * Errors: TK_E_ARG, TK_E_LIMIT (n_bytes or S above the workspace's limits),
 * TK_E_UTF8 (invalid UTF-8; tk_last_error gives the first bad byte offset),
 * TK_E_CAPACITY, TK_E_CUDA, TK_E_TIMEOUT.
 */
int tk_encode_segments(const tk_tokenizer* tok, tk_workspace* ws, const uint8_t* d_text,
                       int64_t n_bytes, const int64_t* d_seg_off,
                       const uint8_t* d_allow_special, int64_t S, int tiktoken_safe,
                       int32_t* d_out_ids, int64_t out_capacity, int64_t* d_out_offsets,
                       int64_t* h_n_ids, void* cuda_stream);

/*
 * tk_encode_segments_host -- the same encode for callers whose data lives in
 * host memory: h_text, h_seg_off, h_allow_special are copied to the
 * workspace's device staging buffers, the encode runs on cuda_stream, and the
 * ids and offsets are copied back into h_out_ids[out_capacity] and
 * h_out_offsets[S+1].  Pinned host buffers make the copies asynchronous.
 * Same arguments and errors as tk_encode_segments.
 */
int tk_encode_segments_host(const tk_tokenizer* tok, tk_workspace* ws, const uint8_t* h_text,
                            int64_t n_bytes, const int64_t* h_seg_off,
                            const uint8_t* h_allow_special, int64_t S, int tiktoken_safe,
                            int32_t* h_out_ids, int64_t out_capacity, int64_t* h_out_offsets,
                            int64_t* h_n_ids, void* cuda_stream);

/*
 * tk_decode -- ids -> bytes on the device ("tiktoken Deep Dive", "The byte
 * floor": a round trip reproduces the input byte for byte; "Pitfalls that
 * bite in production": the output is the concatenated bytes of all ids, since
 * one character's bytes may be spread over several ids).
 *
 *   d_ids[n]: ids (ranks or specials).  d_out[cap]: receives the bytes of each
 *   id in turn.  h_len: the total byte length (also when it exceeds cap, then
 *   TK_E_CAPACITY).  An id that is neither a rank nor a special (for example
 *   one in the reserved gap below the specials) gives TK_E_BADID.
 *   Uses the workspace for scratch (n <= max_bytes).
 */
int tk_decode(const tk_tokenizer* tok, tk_workspace* ws, const int32_t* d_ids, int64_t n,
              uint8_t* d_out, int64_t cap, int64_t* h_len, void* cuda_stream);

/*
 * tk_decode_segments -- tk_decode of S sequences at once (the ids of an
 * encode_segments call, say): d_ids[n] with d_id_off[S+1] (0 = d_id_off[0] <=
 * ... <= d_id_off[S] = n, else TK_E_ARG) -> their bytes one after the other in
 * d_out[cap] and d_byte_off[S+1], the byte offset of each sequence's first
 * byte (d_byte_off[S] = *h_len, the total).  Errors as for tk_decode.
 */
int tk_decode_segments(const tk_tokenizer* tok, tk_workspace* ws, const int32_t* d_ids, int64_t n,
                       const int64_t* d_id_off, int64_t S, uint8_t* d_out, int64_t cap,
                       int64_t* d_byte_off, int64_t* h_len, void* cuda_stream);

/*
 * tk_decode_stream -- incremental decode of ids that arrive in pieces
 * ("tiktoken Deep Dive", "Pitfalls that bite in production": tokens are not
 * characters, so a token can end inside a character; accumulate the bytes and
 * hold back any trailing partial sequence).
 *
 *   state: caller-owned, zeroed before the first call of a stream; holds the
 *       0..3 bytes held back by the previous call.
 *   d_ids[n]: the next ids.  final: nonzero on the last call of the stream
 *       (nothing is held back then; n may be 0 to flush).
 *   d_out[cap]: receives the held-back bytes of the previous call, then the
 *       bytes of d_ids; *h_len = the bytes it may emit now: all of them except
 *       a trailing proper prefix of a well-formed UTF-8 character (a lead byte
 *       C2..F4 with fewer continuation bytes than it announces, the second in
 *       its allowed range), which is kept in state for the next call.  A
 *       surrogate prefix (ED A0..BF) is not held: no character completes it.
 *   cap must hold state->n_pending + the bytes of d_ids; on TK_E_CAPACITY,
 *   *h_len is that total and state is unchanged (the call may be repeated),
 *   as for TK_E_BADID.  Uses the workspace for scratch (n <= max_bytes).
 */
typedef struct tk_decode_state {
  uint8_t pending[4]; /* held-back bytes (n_pending of them) */
  int32_t n_pending;  /* 0..3 */
} tk_decode_state;

int tk_decode_stream(const tk_tokenizer* tok, tk_workspace* ws, tk_decode_state* state,
                     const int32_t* d_ids, int64_t n, int final, uint8_t* d_out, int64_t cap,
                     int64_t* h_len, void* cuda_stream);

/*
 * tk_decode_noalloc -- tk_decode for callers that cannot allocate device
 * memory (a server whose memory pool already holds the device's memory, or a
 * latency-critical path that must not enter the allocator or the device
 * synchronisation cudaFree may imply).  The pages have no counterpart: this
 * is an engineering entry point of this library.
 *
 *   Same arguments and results as tk_decode, without a workspace: d_ids[n]
 *   (n <= 1,048,576, else TK_E_LIMIT), d_out[cap], *h_len = total bytes
 *   (TK_E_CAPACITY when it exceeds cap), TK_E_BADID for an unknown id.
 *   Allocates nothing: its scratch (about 4 KiB of look-back descriptors and
 *   a status block) is a fixed array compiled into the library, held by every
 *   GPU that loads it until the process exits.
 *
 *   The first call on a device looks up that array's device address (with
 *   that device current) and keeps it for the life of the process; make that
 *   first call before any stream capture.  The kept address belongs to the
 *   device's current context: after cudaDeviceReset on that device, do not
 *   call this entry point again in the same process.
 *   All calls on a device share the array: calls that overlap on the GPU race,
 *   so serialise them (for example on one stream).  Each call clears the part
 *   of the array it uses before its kernel runs, then copies its 64-byte
 *   status back into host memory and waits for cuda_stream to finish (every
 *   call synchronises cuda_stream).
 */
int tk_decode_noalloc(const tk_tokenizer* tok, const int32_t* d_ids, int64_t n, uint8_t* d_out,
                      int64_t cap, int64_t* h_len, void* cuda_stream);

/*
 * Cross-call word cache ("Making Kimi K3 Tokenization 18x Faster ...", "Where
 * the speed comes from": repeated words are merged once; "tokenizers v1",
 * "Key Technical Improvements": a word cache).  Within one call every
 * pre-token over 16 bytes is merged once per distinct byte string; a cache
 * keeps those merges between calls, for agent loops that resend most of
 * their prompt.  A hit returns the ids merged earlier for the same bytes and
 * the same tokenizer, so results never change.
 *
 *   tk_cache_create: device memory for max_bytes bytes of cached pieces (and
 *       as many ids, plus an index); nothing is evicted: once full, new
 *       pieces are merged but not added.  The cache belongs to tok.
 *   tk_workspace_set_cache: encodes on ws look pieces up in cache (before
 *       merging) and add the ones they merged (after); NULL detaches.  Encodes
 *       that share a cache must not overlap in time.
 *   tk_cache_clear: empties it (on cuda_stream).  tk_cache_stats: entries,
 *       bytes and ids held (synchronises the device).
 *   tk_last_cache_stats: pieces the workspace's last encode found in the
 *       cache and added to it.
 */
typedef struct tk_cache tk_cache;
int tk_cache_create(const tk_tokenizer* tok, int64_t max_bytes, tk_cache** out);
void tk_cache_free(tk_cache* cache);
int tk_cache_clear(tk_cache* cache, void* cuda_stream);
int tk_cache_stats(const tk_cache* cache, int64_t* n_entries, int64_t* bytes_used, int64_t* ids_used);
int tk_workspace_set_cache(tk_workspace* ws, tk_cache* cache);
int tk_last_cache_stats(const tk_workspace* ws, int64_t* hits, int64_t* inserts);

/*
 * Per-kernel timing of encodes on a workspace, for benchmarks.  With
 * profiling on, every kernel launch of tk_encode_segments /
 * tk_encode_segments_host / tk_decode is bracketed by CUDA events recorded on
 * the call's own stream; after each call the elapsed times are added to
 * per-kernel totals.  tk_profile_enable(ws, 1) turns it on and clears the
 * totals; 0 turns it off.  tk_profile_read copies up to max entries (kernel
 * name, total milliseconds, number of launches) and returns how many kernels
 * have entries.  Names are static strings owned by the library.
 */
int tk_profile_enable(tk_workspace* ws, int on);
int tk_profile_read(const tk_workspace* ws, int max, const char** names, double* total_ms,
                    int64_t* launches);

/*
 * Counts of the last completed tk_encode_segments(_host) call on a workspace
 * (host copies, no device access): pre-tokens found by the split, ids
 * produced, and pre-tokens that took the long-piece merge.  Any pointer may be
 * NULL.
 */
int tk_last_stats(const tk_workspace* ws, int64_t* n_pretokens, int64_t* n_ids, int64_t* n_long);

/* Number of mergeable ranks, specials, and the largest id of a tokenizer. */
int64_t tk_n_ranks(const tk_tokenizer* tok);
int64_t tk_n_specials(const tk_tokenizer* tok);
int64_t tk_max_id(const tk_tokenizer* tok);

/* Static description of a status code, and the calling thread's last error. */
const char* tk_status_string(int code);
const char* tk_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* TK_H */
