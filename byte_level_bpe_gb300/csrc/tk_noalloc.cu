// tk_noalloc.cu -- tk_decode_noalloc: ids -> bytes without allocating.
//
// Some callers cannot call cudaMalloc: a serving process whose memory pool has
// already reserved the device's memory, code on a latency-critical path where
// the allocator (and the device synchronisation cudaFree can imply) is not
// acceptable, or a caller that simply has no workspace at hand when it needs
// to turn a few ids back into text.  This entry point serves them: it reads
// the ids, writes the bytes, and keeps its only scratch (look-back
// descriptors and a status block) in a fixed array compiled into the library.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds its NOALLOC_SCRATCH_BYTES until the process exits, and every
// call on a device shares it.  Calls that overlap on one device therefore
// race (serialise them, e.g. on one stream).  Each call clears the part that
// must start at zero before its kernel runs.
#include <stddef.h>

#include <algorithm>
#include <mutex>

#include "tk_internal.cuh"

namespace tk {

constexpr int64_t NOALLOC_MAX_IDS = 1 << 20;  // ids per call
constexpr int NA_THREADS = 256;
constexpr int NA_ITEMS = 8;
constexpr int64_t NA_TILE = NA_THREADS * NA_ITEMS;
constexpr int64_t NA_MAX_TILES = NOALLOC_MAX_IDS / NA_TILE;

// Status block at the start of the scratch (its first two fields have the
// layout of Status, so the shared look-back can report a timeout into it).
// All zero means "no error, nothing decoded yet".
struct NoAllocStatus {
  int32_t code;        // TK_E_BADID or TK_E_TIMEOUT, 0 if none
  int32_t err_kind;
  int64_t bad_key;     // INT64_MAX - (smallest index of a bad id), 0 if none
  int64_t total;       // bytes of the decoded text
  uint32_t tile_ctr;   // dynamic tile counter
  uint32_t pad;
  uint64_t pad2[4];
};
static_assert(offsetof(NoAllocStatus, code) == offsetof(Status, code) &&
                  offsetof(NoAllocStatus, err_kind) == offsetof(Status, err_kind),
              "status layout shared with the look-back helper");

// the status block, then one look-back descriptor per tile
constexpr size_t NOALLOC_SCRATCH_BYTES = sizeof(NoAllocStatus) + sizeof(uint64_t) * NA_MAX_TILES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

// One pass: each tile of 2,048 ids finds its byte lengths, its byte offset by
// decoupled look-back over the tiles before it, and copies the bytes.
__global__ void __launch_bounds__(NA_THREADS)
k_decode_noalloc(Tables T, const int32_t* __restrict__ ids, int64_t n, uint8_t* __restrict__ out,
                 int64_t cap, unsigned char* scratch) {
  NoAllocStatus* st = reinterpret_cast<NoAllocStatus*>(scratch);
  uint64_t* desc = reinterpret_cast<uint64_t*>(scratch + sizeof(NoAllocStatus));
  __shared__ uint64_t s_warp[NA_THREADS / 32];
  __shared__ int64_t s_tile;
  __shared__ uint64_t s_base;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t ntiles = (n + NA_TILE - 1) / NA_TILE;
  for (;;) {
    if (tid == 0) s_tile = atomicAdd(&st->tile_ctr, 1u);
    __syncthreads();
    const int64_t tile = s_tile;
    if (tile >= ntiles) break;
    const int64_t base_i = tile * NA_TILE + (int64_t)tid * NA_ITEMS;
    int32_t len[NA_ITEMS];
    uint64_t sum = 0;
#pragma unroll
    for (int k = 0; k < NA_ITEMS; k++) {
      const int64_t i = base_i + k;
      int32_t l = 0;
      if (i < n) {
        const int32_t id = ids[i];
        l = (id >= 0 && id <= T.max_id) ? T.tok_len[id] : -1;
        if (l < 0) {
          atomicCAS(&st->code, 0, TK_E_BADID);
          atomicMax((long long*)&st->bad_key, (long long)(INT64_MAX - i));
          l = 0;
        }
      }
      len[k] = l;
      sum += (uint64_t)l;
    }
    // block exclusive scan of the per-thread byte counts
    uint64_t x = sum;
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
      uint64_t run = 0;
      if (lane == 0)
        for (int w = 0; w < NA_THREADS / 32; w++) {
          const uint64_t a = s_warp[w];
          s_warp[w] = run;
          run += a;
        }
      run = __shfl_sync(0xffffffffu, run, 0);
      const uint64_t b = chain_exclusive_warp<SumOp>(desc, tile, run, reinterpret_cast<Status*>(st), 30);
      if (lane == 0) {
        s_base = b;
        if (tile == ntiles - 1) st->total = (int64_t)(b + run);
      }
    }
    __syncthreads();
    uint64_t o = s_base + s_warp[warp] + x - sum;
#pragma unroll
    for (int k = 0; k < NA_ITEMS; k++) {
      const int64_t i = base_i + k;
      if (i < n && len[k] > 0) {
        const uint8_t* src = T.tok_bytes + T.tok_start[ids[i]];
        for (int j = 0; j < len[k]; j++)
          if ((int64_t)(o + j) < cap) out[o + j] = src[j];
      }
      o += (uint64_t)len[k];
    }
    __syncthreads();
  }
}

}  // namespace tk

// Per-device address of the scratch array, resolved once with that device
// current (a __device__ symbol's host-side name is not a device address).
static std::mutex g_noalloc_mutex;
static unsigned char* g_noalloc_ptr[256];

extern "C" int tk_decode_noalloc(const tk_tokenizer* tok, const int32_t* d_ids, int64_t n,
                                 uint8_t* d_out, int64_t cap, int64_t* h_len, void* cuda_stream) {
  using namespace tk;
  if (!tok || n < 0 || cap < 0 || (n > 0 && !d_ids) || (cap > 0 && !d_out)) {
    tk_set_error("tk_decode_noalloc: bad argument");
    return TK_E_ARG;
  }
  if (n > NOALLOC_MAX_IDS) {
    tk_set_error("tk_decode_noalloc: %lld ids above the fixed limit of %lld per call (use tk_decode)",
                 (long long)n, (long long)NOALLOC_MAX_IDS);
    return TK_E_LIMIT;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 256) {
    tk_set_error("tk_decode_noalloc: no current CUDA device");
    return TK_E_CUDA;
  }
  if (dev != tok->device) {
    tk_set_error("tk_decode_noalloc: current device %d is not the tokenizer's device %d", dev, tok->device);
    return TK_E_ARG;
  }
  unsigned char* scratch;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess || !p) {
        tk_set_error("tk_decode_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        return TK_E_CUDA;
      }
      g_noalloc_ptr[dev] = static_cast<unsigned char*>(p);
    }
    scratch = g_noalloc_ptr[dev];
  }
  cudaStream_t st = (cudaStream_t)cuda_stream;
  const int64_t ntiles = (n + NA_TILE - 1) / NA_TILE;
  // clear the status block and the descriptors this call uses
  e = cudaMemsetAsync(scratch, 0, sizeof(NoAllocStatus) + sizeof(uint64_t) * (size_t)ntiles, st);
  if (e == cudaSuccess && n > 0) {
    int sms = 1;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int grid = (int)std::min<int64_t>(ntiles, (int64_t)sms * 4);
    k_decode_noalloc<<<grid, NA_THREADS, 0, st>>>(tok->t, d_ids, n, d_out, cap, scratch);
    e = cudaGetLastError();
  }
  NoAllocStatus res = {};
  if (e == cudaSuccess) e = cudaMemcpyAsync(&res, scratch, sizeof(res), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) {
    tk_set_error("tk_decode_noalloc: %s", cudaGetErrorString(e));
    return TK_E_CUDA;
  }
  if (h_len) *h_len = res.total;
  if (res.code == TK_E_BADID) {
    tk_set_error("tk_decode_noalloc: unknown id at index %lld", (long long)(INT64_MAX - res.bad_key));
    return TK_E_BADID;
  }
  if (res.code) {
    tk_set_error("tk_decode_noalloc: device error %d", res.code);
    return res.code;
  }
  if (res.total > cap) {
    tk_set_error("tk_decode_noalloc: capacity %lld < %lld bytes", (long long)cap, (long long)res.total);
    return TK_E_CAPACITY;
  }
  return TK_OK;
}
