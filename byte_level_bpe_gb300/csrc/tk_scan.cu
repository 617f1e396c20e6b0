// tk_scan.cu -- exclusive scan of u32 counts in one pass (decoupled look-back).
//
// Used for the ordered assembly of ids ("Making Kimi K3 Tokenization 18x
// Faster ...", "Where the speed comes from": output order is restored after
// the per-piece work) and for decode offsets.  The element count is read on
// the device (it is produced by an earlier kernel), so the grid is persistent
// and takes tiles from a counter in the status block.
#include <string.h>

#include <algorithm>

#include "tk_internal.cuh"

namespace tk {

__global__ void __launch_bounds__(SCAN_THREADS)
k_scan_u32(const uint32_t* __restrict__ in, uint32_t* __restrict__ out, const int64_t* d_n,
           uint64_t* desc, Status* st, int ctr) {
  __shared__ uint32_t s_warp[SCAN_THREADS / 32];
  __shared__ int64_t s_tile;
  __shared__ uint64_t s_prefix;
  const int64_t n = *d_n;
  const int64_t ntiles = (n + SCAN_TILE - 1) / SCAN_TILE;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (n == 0) {
    if (blockIdx.x == 0 && tid == 0) out[0] = 0;
    return;
  }
  for (;;) {
    if (tid == 0) s_tile = atomicAdd(&st->tile_ctr[ctr], 1u);
    __syncthreads();
    const int64_t tile = s_tile;
    if (tile >= ntiles) break;
    const int64_t base = tile * SCAN_TILE + (int64_t)tid * SCAN_ITEMS;
    uint32_t v[SCAN_ITEMS];
    uint32_t sum = 0;
#pragma unroll
    for (int i = 0; i < SCAN_ITEMS; i++) {
      v[i] = (base + i < n) ? in[base + i] : 0u;
      sum += v[i];
    }
    // block-wide exclusive scan of the per-thread sums
    uint32_t x = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
      uint32_t w = (lane < SCAN_THREADS / 32) ? s_warp[lane] : 0u;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      if (lane < SCAN_THREADS / 32) s_warp[lane] = w;
    }
    __syncthreads();
    const uint32_t tile_total = s_warp[SCAN_THREADS / 32 - 1];
    const uint32_t excl = (warp ? s_warp[warp - 1] : 0u) + x - sum;
    if (warp == 0) {
      const uint64_t prefix = chain_exclusive_warp<SumOp>(desc, tile, tile_total, st, 10 + ctr);
      if (lane == 0) s_prefix = prefix;
    }
    __syncthreads();
    uint32_t run = (uint32_t)s_prefix + excl;
#pragma unroll
    for (int i = 0; i < SCAN_ITEMS; i++) {
      if (base + i < n) out[base + i] = run;
      run += v[i];
    }
    if (tile == ntiles - 1 && tid == SCAN_THREADS - 1) out[n] = run;
    __syncthreads();
  }
}

}  // namespace tk

int tk_scan_u32(tk_workspace* ws, const uint32_t* d_in, uint32_t* d_out, const int64_t* d_n,
                int64_t n_max, int chain_ctr, cudaStream_t st) {
  const int64_t tiles = (n_max + tk::SCAN_TILE - 1) / tk::SCAN_TILE;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(tiles, (int64_t)ws->num_sms * 8));
  tk::k_scan_u32<<<grid, tk::SCAN_THREADS, 0, st>>>(d_in, d_out, d_n, ws->w.desc_c, ws->w.status,
                                                     chain_ctr);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    tk_set_error("scan launch: %s", cudaGetErrorString(e));
    return TK_E_CUDA;
  }
  return TK_OK;
}

// ---------------------------------------------------------------------------
// Per-kernel profiling with CUDA events on the launching stream.

void tk_prof_mark(tk_workspace* ws, const char* kernel, cudaStream_t st) {
  tk_profile& p = ws->prof;
  if (!p.on || p.n_pending >= tk_profile::MAXK) return;
  cudaEventRecord(p.ev[p.n_pending], st);
  p.pstream[p.n_pending] = st;
  p.pending[p.n_pending++] = kernel;
}

void tk_prof_finish(tk_workspace* ws, cudaStream_t st) {
  tk_profile& p = ws->prof;
  if (!p.on || p.n_pending == 0) return;
  (void)st;
  for (int i = 0; i < p.n_pending; i++) cudaEventSynchronize(p.ev[i]);
  for (int i = 0; i < p.n_pending; i++) {
    if (!p.pending[i]) continue;  // an end mark
    int j = i + 1;
    while (j < p.n_pending && p.pstream[j] != p.pstream[i]) j++;
    if (j == p.n_pending) continue;  // no end mark on that stream
    float ms = 0.f;
    cudaEventElapsedTime(&ms, p.ev[i], p.ev[j]);
    int k = 0;
    while (k < p.n && strcmp(p.names[k], p.pending[i]) != 0) k++;
    if (k == p.n) {
      if (p.n >= tk_profile::MAXK) continue;
      p.names[p.n] = p.pending[i];
      p.total_ms[p.n] = 0;
      p.launches[p.n] = 0;
      p.n++;
    }
    p.total_ms[k] += ms;
    p.launches[k] += 1;
  }
  p.n_pending = 0;
}

extern "C" int tk_profile_enable(tk_workspace* ws, int on) {
  if (!ws) return TK_E_ARG;
  tk_profile& p = ws->prof;
  if (on && !p.ev[0]) {
    for (int i = 0; i <= tk_profile::MAXK; i++)
      if (cudaEventCreate(&p.ev[i]) != cudaSuccess) return TK_E_CUDA;
  }
  p.on = on ? 1 : 0;
  p.n = 0;
  p.n_pending = 0;
  return TK_OK;
}

extern "C" int tk_profile_read(const tk_workspace* ws, int max, const char** names, double* total_ms,
                               int64_t* launches) {
  if (!ws) return TK_E_ARG;
  const tk_profile& p = ws->prof;
  for (int i = 0; i < p.n && i < max; i++) {
    if (names) names[i] = p.names[i];
    if (total_ms) total_ms[i] = p.total_ms[i];
    if (launches) launches[i] = p.launches[i];
  }
  return p.n;
}
