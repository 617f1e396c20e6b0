// tk_tokenizer.cu -- tk_load (table checks and device tables), decode, errors.
//
// An encoding is a bytes -> rank table whose rank is the token id, a split
// pattern and a dict of specials ("tiktoken Deep Dive", "An encoding is three
// objects, not a model").  Loading builds, once, the device tables the
// kernels read:
//   * byte_id[256]: the id of every single byte ("The byte floor");
//   * dense[65536]: the rank of every two-byte token (the first merge round of
//     every pre-token reads this table instead of the hash table);
//   * pair slots: for every token t and every split t = a || b where a and b
//     are tokens, (id(a), id(b)) -> rank(t).  Pieces in the merge loop are
//     always tokens, so "rank of the concatenation of two adjacent pieces" is
//     exactly this lookup on their ids;
//   * specials and their first bytes; the id -> bytes table for decode.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <new>
#include <string>
#include <string_view>
#include <unordered_map>
#include <vector>

#include "tk_internal.cuh"

static thread_local char g_err[512];

void tk_set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

extern "C" const char* tk_last_error(void) { return g_err; }

extern "C" const char* tk_status_string(int code) {
  switch (code) {
    case TK_OK: return "ok";
    case TK_E_ARG: return "bad argument";
    case TK_E_TABLE: return "table rejected";
    case TK_E_UTF8: return "invalid UTF-8";
    case TK_E_CAPACITY: return "output capacity too small";
    case TK_E_CUDA: return "CUDA error";
    case TK_E_NOMEM: return "out of memory";
    case TK_E_TIMEOUT: return "device wait timed out";
    case TK_E_BADID: return "unknown token id";
    case TK_E_LIMIT: return "input above workspace limits";
    default: return "unknown status";
  }
}

static bool valid_utf8(const uint8_t* s, int64_t n) {
  int64_t i = 0;
  while (i < n) {
    const uint8_t b = s[i];
    int len;
    uint32_t c;
    if (b < 0x80) { len = 1; c = b; }
    else if (b >= 0xC2 && b <= 0xDF) { len = 2; c = b & 0x1F; }
    else if (b >= 0xE0 && b <= 0xEF) { len = 3; c = b & 0x0F; }
    else if (b >= 0xF0 && b <= 0xF4) { len = 4; c = b & 0x07; }
    else return false;
    if (i + len > n) return false;
    for (int j = 1; j < len; j++) {
      if ((s[i + j] & 0xC0) != 0x80) return false;
      c = (c << 6) | (s[i + j] & 0x3F);
    }
    if ((len == 3 && (c < 0x800 || (c >= 0xD800 && c <= 0xDFFF))) || (len == 4 && (c < 0x10000 || c > 0x10FFFF)))
      return false;
    i += len;
  }
  return true;
}

template <class T>
static int upload(tk_tokenizer* tk_, const T* src, size_t count, const T** dst) {
  void* p = nullptr;
  const size_t bytes = std::max<size_t>(1, sizeof(T) * count);
  cudaError_t e = cudaMalloc(&p, bytes);
  if (e != cudaSuccess) {
    tk_set_error("tk_load: cudaMalloc(%zu): %s", bytes, cudaGetErrorString(e));
    return TK_E_NOMEM;
  }
  if (tk_->n_dev >= tk_tokenizer::MAX_DEV) {
    cudaFree(p);
    tk_set_error("tk_load: too many device tables");
    return TK_E_NOMEM;
  }
  tk_->dev_mem[tk_->n_dev++] = p;
  if (count) {
    e = cudaMemcpy(p, src, sizeof(T) * count, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
      tk_set_error("tk_load: cudaMemcpy: %s", cudaGetErrorString(e));
      return TK_E_CUDA;
    }
  }
  *dst = static_cast<const T*>(p);
  return TK_OK;
}

extern "C" void tk_free(tk_tokenizer* tok) {
  if (!tok) return;
  for (int i = 0; i < tok->n_dev; i++) cudaFree(tok->dev_mem[i]);
  delete tok;
}

static int table_error(const char* msg, long long a = 0) {
  tk_set_error(msg, a);
  return TK_E_TABLE;
}

extern "C" int tk_load(const uint8_t* rank_bytes, const int64_t* rank_off, const uint32_t* rank_ids,
                       int64_t n, const uint8_t* spec_bytes, const int64_t* spec_off,
                       const int32_t* spec_ids, int64_t n_spec, int pattern_id, tk_tokenizer** out) {
  using namespace tk;
  if (!out) return TK_E_ARG;
  *out = nullptr;
  if (pattern_id != TK_PATTERN_CL100K && pattern_id != TK_PATTERN_R50K_DIGITS) {
    tk_set_error("tk_load: unknown pattern_id %d", pattern_id);
    return TK_E_ARG;
  }
  if (n <= 0 || !rank_bytes || !rank_off || !rank_ids || n_spec < 0 || (n_spec > 0 && (!spec_bytes || !spec_off || !spec_ids))) {
    tk_set_error("tk_load: bad argument");
    return TK_E_ARG;
  }
  if (rank_off[0] != 0 || (n_spec > 0 && spec_off[0] != 0)) {
    tk_set_error("tk_load: offsets must start at 0");
    return TK_E_ARG;
  }
  if (n_spec > MAX_SPECIALS) return table_error("tk_load: more than %lld specials", MAX_SPECIALS);
  // ---- ranks
  std::unordered_map<std::string_view, uint32_t> by_bytes;
  by_bytes.reserve((size_t)n * 2);
  int64_t max_id = -1;
  for (int64_t i = 0; i < n; i++) {
    const int64_t len = rank_off[i + 1] - rank_off[i];
    if (len <= 0) return table_error("tk_load: empty token at index %lld", (long long)i);
    if (rank_ids[i] > MAX_ID) return table_error("tk_load: id %lld too large", (long long)rank_ids[i]);
    std::string_view key(reinterpret_cast<const char*>(rank_bytes + rank_off[i]), (size_t)len);
    if (!by_bytes.emplace(key, rank_ids[i]).second)
      return table_error("tk_load: duplicate token bytes at index %lld", (long long)i);
    max_id = std::max<int64_t>(max_id, rank_ids[i]);
  }
  uint32_t byte_id[256];
  for (int b = 0; b < 256; b++) {
    const char ch = (char)b;
    auto it = by_bytes.find(std::string_view(&ch, 1));
    if (it == by_bytes.end()) return table_error("tk_load: byte %lld is not a token (byte floor)", b);
    byte_id[b] = it->second;
  }
  // ---- specials
  for (int64_t i = 0; i < n_spec; i++) {
    const int64_t len = spec_off[i + 1] - spec_off[i];
    if (len <= 0 || len > MAX_SPECIAL) return table_error("tk_load: special %lld is empty or longer than 64 bytes", (long long)i);
    if (!valid_utf8(spec_bytes + spec_off[i], len)) return table_error("tk_load: special %lld is not valid UTF-8", (long long)i);
    if (spec_ids[i] < 0 || spec_ids[i] > (int32_t)MAX_ID) return table_error("tk_load: special id %lld out of range", spec_ids[i]);
    max_id = std::max<int64_t>(max_id, spec_ids[i]);
  }
  std::vector<int8_t> used((size_t)max_id + 1, 0);
  for (int64_t i = 0; i < n; i++) {
    if (used[rank_ids[i]]) return table_error("tk_load: duplicate id %lld", (long long)rank_ids[i]);
    used[rank_ids[i]] = 1;
  }
  for (int64_t i = 0; i < n_spec; i++) {
    if (used[spec_ids[i]]) return table_error("tk_load: special id %lld collides with another id", spec_ids[i]);
    used[spec_ids[i]] = 2;
  }
  // specials must not overlap in text: no proper suffix of one is a prefix of
  // another (or contains it), so every match found is taken
  for (int64_t a = 0; a < n_spec; a++) {
    const uint8_t* A = spec_bytes + spec_off[a];
    const int64_t la = spec_off[a + 1] - spec_off[a];
    for (int64_t b = 0; b < n_spec; b++) {
      const uint8_t* B = spec_bytes + spec_off[b];
      const int64_t lb = spec_off[b + 1] - spec_off[b];
      for (int64_t k = 1; k < la; k++) {
        const int64_t m = std::min<int64_t>(la - k, lb);
        if (memcmp(A + k, B, (size_t)m) == 0)
          return table_error("tk_load: specials %lld and another can overlap in text", (long long)a);
      }
    }
  }
  // ---- merge tables
  std::vector<uint32_t> dense(65536, RANK_MAX);
  std::vector<std::pair<uint64_t, uint32_t>> pairs;
  pairs.reserve((size_t)n * 2);
  for (int64_t i = 0; i < n; i++) {
    const int64_t len = rank_off[i + 1] - rank_off[i];
    const char* p = reinterpret_cast<const char*>(rank_bytes + rank_off[i]);
    if (len == 2) dense[((uint8_t)p[0] << 8) | (uint8_t)p[1]] = rank_ids[i];
    for (int64_t k = 1; k < len; k++) {
      auto a = by_bytes.find(std::string_view(p, (size_t)k));
      if (a == by_bytes.end()) continue;
      auto b = by_bytes.find(std::string_view(p + k, (size_t)(len - k)));
      if (b == by_bytes.end()) continue;
      pairs.emplace_back(((uint64_t)a->second << 20) | b->second, rank_ids[i]);
    }
  }
  // tokens with an extension that ranks below them: only a merge into such a
  // token can create a neighbour pair below the round's rank
  std::vector<uint8_t> ext_low((size_t)max_id + 1, 0);
  for (auto& kv : pairs) {
    const uint32_t a = (uint32_t)(kv.first >> 20), b = (uint32_t)(kv.first & 0xFFFFF);
    if (kv.second < b) ext_low[b] |= 1;
    if (kv.second < a) ext_low[a] |= 2;
  }
  uint32_t log2cap = 10;
  while ((1ull << log2cap) < 2 * pairs.size() + 16) log2cap++;
  std::vector<uint64_t> slots(1ull << log2cap, ~0ull);
  uint32_t max_probe = 0;
  const uint64_t mask = (1ull << log2cap) - 1;
  for (auto& kv : pairs) {
    uint64_t h = (kv.first * 0x9E3779B97F4A7C15ull) >> (64 - log2cap);
    uint32_t probe = 0;
    while (slots[h] != ~0ull) { h = (h + 1) & mask; probe++; }
    slots[h] = (kv.first << 20) | kv.second;
    max_probe = std::max(max_probe, probe);
  }
  // slice table of the 3- and 4-byte tokens (one probe, independent of the
  // pair ranks, gives a three- or four-byte piece its longer slices)
  std::vector<uint64_t> s34_items;
  for (int64_t i = 0; i < n; i++) {
    const int64_t len = rank_off[i + 1] - rank_off[i];
    if (len != 3 && len != 4) continue;
    const uint8_t* p = rank_bytes + rank_off[i];
    const uint32_t key = p[0] | (uint32_t)p[1] << 8 | (uint32_t)p[2] << 16 | (len == 4 ? (uint32_t)p[3] << 24 : 0u);
    s34_items.push_back(((uint64_t)key << 21) | ((uint64_t)(len == 4) << 20) | rank_ids[i]);
  }
  uint32_t s34_log2 = 10;
  while ((1ull << s34_log2) < 4 * s34_items.size() + 16) s34_log2++;
  std::vector<uint64_t> s34(1ull << s34_log2, ~0ull);
  uint32_t s34_max_probe = 0;
  for (uint64_t it : s34_items) {
    uint32_t h = s34_hash((uint32_t)(it >> 21), s34_log2);
    uint32_t probe = 0;
    while (s34[h] != ~0ull) { h = (h + 1) & (uint32_t)((1ull << s34_log2) - 1); probe++; }
    s34[h] = it;
    s34_max_probe = std::max(s34_max_probe, probe);
  }
  // ---- decode table
  std::vector<uint32_t> tok_start((size_t)max_id + 1, 0);
  std::vector<int32_t> tok_len((size_t)max_id + 1, -1);
  std::vector<uint8_t> tok_bytes;
  tok_bytes.reserve((size_t)rank_off[n] + (n_spec ? (size_t)spec_off[n_spec] : 0));
  for (int64_t i = 0; i < n; i++) {
    tok_start[rank_ids[i]] = (uint32_t)tok_bytes.size();
    tok_len[rank_ids[i]] = (int32_t)(rank_off[i + 1] - rank_off[i]);
    tok_bytes.insert(tok_bytes.end(), rank_bytes + rank_off[i], rank_bytes + rank_off[i + 1]);
  }
  std::vector<int32_t> soff(n_spec + 1, 0), sid(std::max<int64_t>(n_spec, 1), 0);
  std::vector<uint8_t> sbytes;
  Tables t = {};
  for (int64_t i = 0; i < n_spec; i++) {
    tok_start[spec_ids[i]] = (uint32_t)tok_bytes.size();
    tok_len[spec_ids[i]] = (int32_t)(spec_off[i + 1] - spec_off[i]);
    tok_bytes.insert(tok_bytes.end(), spec_bytes + spec_off[i], spec_bytes + spec_off[i + 1]);
    sbytes.insert(sbytes.end(), spec_bytes + spec_off[i], spec_bytes + spec_off[i + 1]);
    soff[i + 1] = (int32_t)sbytes.size();
    sid[i] = spec_ids[i];
    const uint8_t f = spec_bytes[spec_off[i]];
    t.spec_first[f >> 5] |= 1u << (f & 31);
  }
  // ---- device
  tk_tokenizer* tok = new (std::nothrow) tk_tokenizer();
  if (!tok) return TK_E_NOMEM;
  cudaError_t e = cudaGetDevice(&tok->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&tok->num_sms, cudaDevAttrMultiProcessorCount, tok->device);
  if (e != cudaSuccess) {
    tk_set_error("tk_load: no CUDA device: %s", cudaGetErrorString(e));
    delete tok;
    return TK_E_CUDA;
  }
  int rc = TK_OK;
  rc = rc ? rc : upload(tok, byte_id, 256, &t.byte_id);
  rc = rc ? rc : upload(tok, dense.data(), dense.size(), &t.dense);
  rc = rc ? rc : upload(tok, slots.data(), slots.size(), &t.pair_slots);
  rc = rc ? rc : upload(tok, ext_low.data(), ext_low.size(), &t.ext_low);
  rc = rc ? rc : upload(tok, s34.data(), s34.size(), &t.s34_slots);
  rc = rc ? rc : upload(tok, sbytes.data(), sbytes.size(), &t.spec_bytes);
  rc = rc ? rc : upload(tok, soff.data(), soff.size(), &t.spec_off);
  rc = rc ? rc : upload(tok, sid.data(), sid.size(), &t.spec_ids);
  rc = rc ? rc : upload(tok, tok_start.data(), tok_start.size(), &t.tok_start);
  rc = rc ? rc : upload(tok, tok_len.data(), tok_len.size(), &t.tok_len);
  rc = rc ? rc : upload(tok, tok_bytes.data(), tok_bytes.size(), &t.tok_bytes);
  if (rc) {
    tk_free(tok);
    return rc;
  }
  t.pattern = pattern_id;
  t.pair_log2 = log2cap;
  t.pair_max_probe = max_probe;
  t.s34_log2 = s34_log2;
  t.s34_max_probe = s34_max_probe;
  t.n_spec = (int32_t)n_spec;
  t.max_id = max_id;
  tok->t = t;
  tok->n_ranks = n;
  *out = tok;
  return TK_OK;
}

extern "C" int64_t tk_n_ranks(const tk_tokenizer* tok) { return tok ? tok->n_ranks : -1; }
extern "C" int64_t tk_n_specials(const tk_tokenizer* tok) { return tok ? tok->t.n_spec : -1; }
extern "C" int64_t tk_max_id(const tk_tokenizer* tok) { return tok ? tok->t.max_id : -1; }

// ---------------------------------------------------------------------------
// Decode: id -> byte length, scan, copy.

namespace tk {

__global__ void k_dec_reset(Work W, int64_t n_desc, int64_t n) {
  const int64_t tid = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (tid == 0) {
    Status s = {};
    s.err_pos = INT64_MAX;
    s.n_ptok = n;  // element count for the scan
    *W.status = s;
  }
  for (int64_t i = tid; i < n_desc; i += (int64_t)gridDim.x * blockDim.x) W.desc_c[i] = 0;
}

__global__ void k_dec_len(Tables T, Work W, const int32_t* ids, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int32_t id = ids[i];
    int32_t len = (id >= 0 && id <= T.max_id) ? T.tok_len[id] : -1;
    if (len < 0) {
      set_error(W.status, TK_E_BADID, 20);
      atomicMin((long long*)&W.status->err_pos, (long long)i);
      len = 0;
    }
    W.cnt[i] = (uint32_t)len;
  }
}

__global__ void k_dec_copy(Tables T, Work W, const int32_t* ids, int64_t n, uint8_t* out, int64_t cap) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const uint32_t o = W.offs[i], len = W.cnt[i];
    if (len == 0) continue;
    const uint8_t* src = T.tok_bytes + T.tok_start[ids[i]];
    for (uint32_t j = 0; j < len; j++)
      if ((int64_t)o + j < cap) out[o + j] = src[j];
  }
}

__global__ void k_dec_total(Work W, int64_t n) { W.status->n_ids = W.offs[n]; }

}  // namespace tk

// Enqueues a decode of d_ids[n] into d_out[cap] on st (no sync); the byte
// total lands in the status block (n_ids).
static int decode_enqueue(const tk_tokenizer* tok, tk_workspace* ws, const int32_t* d_ids, int64_t n,
                          uint8_t* d_out, int64_t cap, cudaStream_t st) {
  using namespace tk;
  const int64_t n_desc = (n + 1 + SCAN_TILE - 1) / SCAN_TILE + 1;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((n + 255) / 256, (int64_t)ws->num_sms * 8));
  tk_prof_mark(ws, "k_dec_reset", st);
  k_dec_reset<<<ws->num_sms, 256, 0, st>>>(ws->w, n_desc, n);
  if (n > 0) {
    tk_prof_mark(ws, "k_dec_len", st);
    k_dec_len<<<grid, 256, 0, st>>>(tok->t, ws->w, d_ids, n);
  }
  tk_prof_mark(ws, "k_scan_u32", st);
  int rc = tk_scan_u32(ws, ws->w.cnt, ws->w.offs, &ws->w.status->n_ptok, n, 3, st);
  if (rc) return rc;
  if (n > 0) {
    tk_prof_mark(ws, "k_dec_copy", st);
    k_dec_copy<<<grid, 256, 0, st>>>(tok->t, ws->w, d_ids, n, d_out, cap);
  }
  tk_prof_mark(ws, "k_dec_total", st);
  k_dec_total<<<1, 1, 0, st>>>(ws->w, n);
  tk_prof_mark(ws, nullptr, st);
  return TK_OK;
}

// Reads the status back and turns it into a return code (total = bytes needed).
static int decode_finish(tk_workspace* ws, int64_t cap, int64_t extra, cudaStream_t st, const char* who) {
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaMemcpyAsync(ws->h_status, ws->w.status, sizeof(tk::Status), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) {
    tk_set_error("%s: %s", who, cudaGetErrorString(e));
    return TK_E_CUDA;
  }
  tk_prof_finish(ws, st);
  if (ws->h_status->code == TK_E_BADID) {
    tk_set_error("%s: unknown id at index %lld", who, (long long)ws->h_status->err_pos);
    return TK_E_BADID;
  }
  if (ws->h_status->code) {
    tk_set_error("%s: device error %d", who, ws->h_status->code);
    return ws->h_status->code;
  }
  if (ws->h_status->n_ids + extra > cap) {
    tk_set_error("%s: capacity %lld < %lld bytes", who, (long long)cap, (long long)(ws->h_status->n_ids + extra));
    return TK_E_CAPACITY;
  }
  return TK_OK;
}

extern "C" int tk_decode(const tk_tokenizer* tok, tk_workspace* ws, const int32_t* d_ids, int64_t n,
                         uint8_t* d_out, int64_t cap, int64_t* h_len, void* cuda_stream) {
  using namespace tk;
  if (!tok || !ws || n < 0 || cap < 0 || (n > 0 && !d_ids) || (cap > 0 && !d_out)) {
    tk_set_error("tk_decode: bad argument");
    return TK_E_ARG;
  }
  if (n > ws->w.max_bytes) {
    tk_set_error("tk_decode: %lld ids above the workspace limit %lld", (long long)n, (long long)ws->w.max_bytes);
    return TK_E_LIMIT;
  }
  cudaSetDevice(ws->device);
  cudaStream_t st = (cudaStream_t)cuda_stream;
  int rc = decode_enqueue(tok, ws, d_ids, n, d_out, cap, st);
  if (rc) return rc;
  rc = decode_finish(ws, cap, 0, st, "tk_decode");
  if (h_len) *h_len = ws->h_status->n_ids;
  return rc;
}

namespace tk {
// byte_off[s] = bytes before segment s's first id (the decode's exclusive scan
// at id_off[s]); the id offsets must run 0 = id_off[0] <= ... <= id_off[S] = n.
__global__ void k_dec_seg_offsets(Work W, const int64_t* id_off, int64_t S, int64_t n, int64_t* byte_off) {
  for (int64_t s = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; s <= S; s += (int64_t)gridDim.x * blockDim.x) {
    const int64_t a = id_off[s];
    const bool ok = a >= 0 && a <= n && (s > 0 || a == 0) && (s < S || a == n) && (s == S || id_off[s + 1] >= a);
    if (!ok) {
      set_error(W.status, TK_E_ARG, 21);
      continue;
    }
    byte_off[s] = W.offs[a];
  }
}

// How many bytes at the end of b[0..n) start a character that is not complete
// yet: step back over at most three continuation bytes (10xxxxxx) to the
// character's first byte; if that byte announces more bytes than are present
// (C2..DF: 2, E0..EF: 3, F0..F4: 4) and the second byte, if present, is in its
// well-formed range (E0: A0..BF, ED: 80..9F, F0: 90..BF, F4: 80..8F), all of
// them wait for the next call.
__device__ int utf8_partial_tail(const uint8_t* b, int64_t n) {
  int64_t p = n - 1;
  int back = 0;
  while (p >= 0 && back < 3 && (b[p] & 0xC0u) == 0x80u) {
    p--;
    back++;
  }
  if (p < 0) return 0;
  const uint32_t lead = b[p];
  const int want = (lead >= 0xC2u && lead <= 0xDFu) ? 2 : (lead >= 0xE0u && lead <= 0xEFu) ? 3
                 : (lead >= 0xF0u && lead <= 0xF4u) ? 4 : 0;
  const int have = (int)(n - p);
  if (want == 0 || have >= want) return 0;
  if (have >= 2) {
    const uint32_t s = b[p + 1];
    const uint32_t lo = lead == 0xE0u ? 0xA0u : lead == 0xF0u ? 0x90u : 0x80u;
    const uint32_t hi = lead == 0xEDu ? 0x9Fu : lead == 0xF4u ? 0x8Fu : 0xBFu;
    if (s < lo || s > hi) return 0;
  }
  return have;
}

// One thread: the held-back count and bytes of a streaming decode whose
// output holds np pending bytes followed by the decoded ones.
__global__ void k_dec_holdback(Work W, const uint8_t* out, int64_t np, int64_t cap, int final) {
  const int64_t total = np + W.status->n_ids;
  int hb = 0;
  uint32_t tail = 0;
  if (!final && total <= cap && W.status->code == 0) {
    hb = utf8_partial_tail(out, total);
    for (int j = 0; j < hb; j++) tail |= (uint32_t)out[total - hb + j] << (8 * j);
  }
  W.status->holdback = hb;
  W.status->tail = tail;
}
}  // namespace tk

extern "C" int tk_decode_stream(const tk_tokenizer* tok, tk_workspace* ws, tk_decode_state* state,
                                const int32_t* d_ids, int64_t n, int final, uint8_t* d_out, int64_t cap,
                                int64_t* h_len, void* cuda_stream) {
  using namespace tk;
  if (!tok || !ws || !state || n < 0 || cap < 0 || (n > 0 && !d_ids) || (cap > 0 && !d_out) ||
      state->n_pending < 0 || state->n_pending > 3) {
    tk_set_error("tk_decode_stream: bad argument");
    return TK_E_ARG;
  }
  if (n > ws->w.max_bytes) {
    tk_set_error("tk_decode_stream: %lld ids above the workspace limit %lld", (long long)n,
                 (long long)ws->w.max_bytes);
    return TK_E_LIMIT;
  }
  cudaSetDevice(ws->device);
  cudaStream_t st = (cudaStream_t)cuda_stream;
  const int64_t np = state->n_pending;
  const bool fits = cap >= np;  // else only the total is computed (TK_E_CAPACITY)
  if (np && fits) {
    // the held-back bytes go first (a copy from pageable memory: the runtime
    // has taken the bytes when the call returns)
    uint8_t pend[4];
    memcpy(pend, state->pending, (size_t)np);
    const cudaError_t e = cudaMemcpyAsync(d_out, pend, (size_t)np, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) {
      tk_set_error("tk_decode_stream: pending bytes: %s", cudaGetErrorString(e));
      return TK_E_CUDA;
    }
  }
  int rc = decode_enqueue(tok, ws, d_ids, n, fits ? d_out + np : nullptr, fits ? cap - np : 0, st);
  if (rc) return rc;
  k_dec_holdback<<<1, 1, 0, st>>>(ws->w, d_out, np, cap, final ? 1 : 0);
  rc = decode_finish(ws, cap, np, st, "tk_decode_stream");
  const int64_t total = np + ws->h_status->n_ids;
  if (rc) {
    if (h_len) *h_len = total;
    return rc;  // the state is unchanged: the call may be repeated
  }
  const int hb = ws->h_status->holdback;
  for (int j = 0; j < 4; j++) state->pending[j] = j < hb ? (uint8_t)(ws->h_status->tail >> (8 * j)) : 0;
  state->n_pending = hb;
  if (h_len) *h_len = total - hb;
  return TK_OK;
}

extern "C" int tk_decode_segments(const tk_tokenizer* tok, tk_workspace* ws, const int32_t* d_ids, int64_t n,
                                  const int64_t* d_id_off, int64_t S, uint8_t* d_out, int64_t cap,
                                  int64_t* d_byte_off, int64_t* h_len, void* cuda_stream) {
  using namespace tk;
  if (!tok || !ws || n < 0 || S < 0 || cap < 0 || (n > 0 && !d_ids) || (cap > 0 && !d_out) || !d_id_off ||
      !d_byte_off) {
    tk_set_error("tk_decode_segments: bad argument");
    return TK_E_ARG;
  }
  if (n > ws->w.max_bytes) {
    tk_set_error("tk_decode_segments: %lld ids above the workspace limit %lld", (long long)n,
                 (long long)ws->w.max_bytes);
    return TK_E_LIMIT;
  }
  cudaSetDevice(ws->device);
  cudaStream_t st = (cudaStream_t)cuda_stream;
  int rc = decode_enqueue(tok, ws, d_ids, n, d_out, cap, st);
  if (rc) return rc;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((S + 256) / 256, (int64_t)ws->num_sms * 4));
  tk_prof_mark(ws, "k_dec_seg_offsets", st);
  k_dec_seg_offsets<<<grid, 256, 0, st>>>(ws->w, d_id_off, S, n, d_byte_off);
  tk_prof_mark(ws, nullptr, st);
  rc = decode_finish(ws, cap, 0, st, "tk_decode_segments");
  if (h_len) *h_len = ws->h_status->n_ids;
  if (rc == TK_E_ARG) tk_set_error("tk_decode_segments: id offsets must run 0 <= ... <= n");
  return rc;
}
