// Gather of the missing K/V rows from pinned host memory into the resident
// HBM slots, in place, without the copy engines.
//
// Method: "ASPLOS'26 | SpeContext 让小模型先圈出重要 KV Cache" (marsggbo blog)
// §4 (the asynchronous prefetcher moves the missing KV from CPU to GPU on a
// second CUDA stream), §6 (only S_now - S_last is moved), §7 (an offloaded
// layer keeps a budget-sized workspace on the GPU); "SpeContext: Enabling
// Efficient Long-context Reasoning with Speculative Context Sparsity in LLMs"
// (paperlayer.ai summary) §5.1, §5.4 (loads performed in place).
//
// GB300 design: the host store is mapped pinned memory read over the
// NVLink-C2C link by ordinary 16-byte loads, laid out position-major
// ([cap][n_kv][layers][2][d]): the GPU translates host addresses page by page
// across the link, and one load (position p, KV head g) is a single
// contiguous run holding the K and V rows of every layer of the launch. One
// warp streams one load's run: each instruction moves one layer's K row
// (lanes 0-15) and V row (lanes 16-31), 512 contiguous bytes, with up to 16
// layers in flight (a whole 16-layer chunk's run in one round trip); the
// (position, slot) pair and the segment search are done once per load. A
// small grid (two warps per SM on average, in CTAs of 4 warps) keeps about 2.5 MB in
// flight, enough for the link, and leaves the rest of the GPU to the
// kernels that run beside the gather on the other streams (attention, key
// scan). The flattened load index maps back to (request, KV head, i) through
// a prefix sum of n_load kept in shared memory.
#include "spc_device.cuh"
#include "spc_internal.h"

#include <algorithm>

namespace spc {

// CTAs of 4 warps (16K registers), two warps per SM on average, i.e. one CTA
// on every other SM. Measured on GB300 (70B-shaped workload, 80 layers, gathers
// of ~380 MB beside the attention kernel; 32K-context workload, gathers of
// ~12 MB beside the key scan): 512-thread CTAs, each needing a whole register
// file and so waiting for an SM to drain, gave 10.8-10.9 ms/step and 130 us/step;
// 128-thread CTAs 9.4-9.6 ms and 150 us; 64-thread CTAs on every SM 9.7-10.1 ms
// and 210 us (host-link loads on every SM slowed the key scan beside them).
#ifndef SPC_GATHER_THREADS
#define SPC_GATHER_THREADS 128
#endif
constexpr int kGatherThreads = SPC_GATHER_THREADS;
#ifndef SPC_GATHER_UNROLL
#define SPC_GATHER_UNROLL 16   // layers of one run in flight per warp (a 16-layer chunk in one round trip)
#endif
constexpr int kGatherUnroll = SPC_GATHER_UNROLL;
constexpr int kGatherMaxSeg = 1024;
#ifndef SPC_GATHER_WARPS_PER_SM
#define SPC_GATHER_WARPS_PER_SM 2   // ~2.5 MB in flight on 152 SMs, enough for the host link
#endif
constexpr int kGatherWarpsPerSm = SPC_GATHER_WARPS_PER_SM;

__global__ void __launch_bounds__(kGatherThreads)
gather_kernel(const spc_gather_view* __restrict__ views, int layer_lo, int layer_hi,
              const int32_t* __restrict__ load_slot, const int32_t* __restrict__ load_pos,
              const int32_t* __restrict__ n_load, int B, int n_kv, int cap, int K) {
  __shared__ int pre[kGatherMaxSeg + 1];
  __shared__ int scratch[33];
  __shared__ spc_gather_view sv[SPC_MAX_BATCH];
  const int nseg = B * n_kv;
  const int tid = threadIdx.x;

  for (int i = tid; i < B; i += kGatherThreads) sv[i] = views[i];
  int run = 0;
  for (int c0 = 0; c0 < nseg; c0 += kGatherThreads) {
    const int v = (c0 + tid < nseg) ? n_load[c0 + tid] : 0;
    int tot;
    const int ex = block_excl_scan(v, scratch, &tot);
    if (c0 + tid < nseg) pre[c0 + tid] = run + ex;
    run += tot;
  }
  if (tid == 0) pre[nseg] = run;
  __syncthreads();

  const int R = run;
  const int lane = tid & 31, piece = lane & 15, kv = lane >> 4;
  const int w0 = (blockIdx.x * kGatherThreads + tid) >> 5;
  const int nw = (gridDim.x * kGatherThreads) >> 5;
  for (int j = w0; j < R; j += nw) {
    // largest seg with pre[seg] <= j (segments with no load have equal bounds)
    int lo = 0, hi = nseg - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= j) lo = mid; else hi = mid - 1;
    }
    const int seg = lo, i = j - pre[seg];
    const int b = seg / n_kv, g = seg - b * n_kv;
    const spc_gather_view vw = sv[b];
    // layers of this launch the request holds in host memory and in its store
    const int l_begin = max(layer_lo, max(vw.layer0, vw.store_layer0));
    const int l_end = min(layer_hi, min(vw.layer0 + vw.n_layers, vw.store_layer0 + vw.store_layers));
    if (l_begin >= l_end) continue;
    const size_t li = (size_t)seg * K + i;
    const int pos = __ldg(load_pos + li);
    const int slot = __ldg(load_slot + li);
    // the run: store[pos, g, l - store_layer0, kv, :] for l in [l_begin, l_end)
    const uint16_t* run = static_cast<const uint16_t*>(vw.host) +
                          (((size_t)pos * n_kv + g) * vw.store_layers + (l_begin - vw.store_layer0)) * 2 * kD +
                          kv * kD + piece * 8;
    uint16_t* dst0 = static_cast<uint16_t*>(vw.slots) +
                     ((((size_t)(l_begin - vw.layer0) * 2 + kv) * n_kv + g) * K + slot) * kD + piece * 8;
    const size_t dst_layer = (size_t)2 * n_kv * K * kD;     // elements between two layers' slots
    for (int l0 = 0; l0 < l_end - l_begin; l0 += kGatherUnroll) {
      uint4 v[kGatherUnroll];
#pragma unroll
      for (int u = 0; u < kGatherUnroll; ++u)
        if (l0 + u < l_end - l_begin) v[u] = ldg_stream(run + (size_t)(l0 + u) * 2 * kD);
#pragma unroll
      for (int u = 0; u < kGatherUnroll; ++u)
        if (l0 + u < l_end - l_begin) stg_v4(dst0 + (size_t)(l0 + u) * dst_layer, v[u]);
    }
  }
}


// Slot fill of layers entering the host ([Blog] §7: an offloaded layer keeps a
// budget-sized workspace on the GPU; it starts out holding the resident rows).
// One 256-byte row per half-warp, grid-stride over (layer, K/V, request, KV
// head, slot); slots whose position is empty or outside [0, cap) are left
// untouched. The source may be device memory (the layer's HBM cache) or a
// device-visible host address.
constexpr int kFillThreads = 256;

__global__ void __launch_bounds__(kFillThreads)
fill_slots_kernel(const spc_gather_view* __restrict__ views, int layer_lo, int layer_hi,
                  const int32_t* __restrict__ slot_pos, int B, int n_kv, int cap, int K) {
  const int l16 = threadIdx.x & 15;
  const long long per_layer = 2LL * B * n_kv * K;
  const long long total = (long long)(layer_hi - layer_lo) * per_layer;
  const long long nhw = (long long)gridDim.x * (kFillThreads / 16);
  for (long long item = ((long long)blockIdx.x * kFillThreads + threadIdx.x) >> 4; item < total; item += nhw) {
    const int lq = (int)(item / per_layer);
    long long rem = item - lq * per_layer;
    const int kv = (int)(rem / ((long long)B * n_kv * K));
    rem -= (long long)kv * B * n_kv * K;
    const int seg = (int)(rem / K), slot = (int)(rem - (long long)seg * K);
    const int b = seg / n_kv, g = seg - b * n_kv;
    const spc_gather_view vw = views[b];
    const int lrel = layer_lo + lq - vw.layer0;
    if (lrel < 0 || lrel >= vw.n_layers) continue;
    const int pos = slot_pos[(size_t)seg * K + slot];
    if (pos < 0 || pos >= cap) continue;
    const size_t hrow = ((((size_t)lrel * 2 + kv) * n_kv + g) * cap + pos) * kD + l16 * 8;
    const size_t srow = ((((size_t)lrel * 2 + kv) * n_kv + g) * K + slot) * kD + l16 * 8;
    const uint4 v = ldg_stream(static_cast<const uint16_t*>(vw.host) + hrow);
    stg_v4(static_cast<uint16_t*>(vw.slots) + srow, v);
  }
}

int fill_slots_launch(const spc_gather_view* views, int layer_lo, int layer_hi, const int32_t* slot_pos,
                      int B, int n_kv, int cap, int budget, void* stream) {
  if (layer_hi <= layer_lo) return SPC_OK;
  const long long items = (long long)(layer_hi - layer_lo) * 2 * B * n_kv * budget;
  long long grid = (items + (kFillThreads / 16) - 1) / (kFillThreads / 16);
  const long long cap_grid = 4LL * std::max(1, device_sm_count());
  if (grid > cap_grid) grid = cap_grid;
  if (grid < 1) grid = 1;
  fill_slots_kernel<<<(int)grid, kFillThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      views, layer_lo, layer_hi, slot_pos, B, n_kv, cap, budget);
  return cudaGetLastError() == cudaSuccess ? SPC_OK : SPC_ERR_CUDA;
}

// One layer of a layer-major cache ([2][n_kv][cap][d], device memory) into a
// position-major host store ([cap][n_kv][store_layers][2][d]): one 256-byte
// row per half-warp, items in store order (position, KV head, K/V) so each
// (position, head) pair is written as one 512-byte run.
__global__ void __launch_bounds__(kFillThreads)
store_layer_kernel(uint16_t* __restrict__ store, const uint16_t* __restrict__ src, int n_kv, int cap, int rows,
                   int store_layers, int layer) {
  const int l16 = threadIdx.x & 15;
  const long long total = (long long)rows * n_kv * 2;
  const long long nhw = (long long)gridDim.x * (kFillThreads / 16);
  for (long long item = ((long long)blockIdx.x * kFillThreads + threadIdx.x) >> 4; item < total; item += nhw) {
    const long long p = item / (2 * n_kv);
    const int rem = (int)(item - p * 2 * n_kv);
    const int g = rem >> 1, kv = rem & 1;
    const uint4 v = ldg_stream(src + (((size_t)kv * n_kv + g) * cap + p) * kD + l16 * 8);
    stg_v4(store + ((((size_t)p * n_kv + g) * store_layers + layer) * 2 + kv) * kD + l16 * 8, v);
  }
}

int store_layer_launch(void* store, const void* src, int n_kv, int cap, int rows, int store_layers, int layer,
                       void* stream) {
  if (rows <= 0) return SPC_OK;
  const long long items = (long long)rows * n_kv * 2;
  long long grid = (items + (kFillThreads / 16) - 1) / (kFillThreads / 16);
  const long long cap_grid = 2LL * std::max(1, device_sm_count());
  if (grid > cap_grid) grid = cap_grid;
  store_layer_kernel<<<(int)grid, kFillThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint16_t*>(store), static_cast<const uint16_t*>(src), n_kv, cap, rows, store_layers, layer);
  return cudaGetLastError() == cudaSuccess ? SPC_OK : SPC_ERR_CUDA;
}

int gather_launch(const spc_gather_view* views, int layer_lo, int layer_hi, const int32_t* load_slot,
                  const int32_t* load_pos, const int32_t* n_load, int B, int n_kv, int cap,
                  int budget, void* stream) {
  if (layer_hi <= layer_lo) return SPC_OK;
  const long long max_loads = (long long)B * n_kv * budget;          // one warp per load at a time
  const long long per_block = kGatherThreads / 32;
  long long grid = (max_loads + per_block - 1) / per_block;
  const long long cap_grid =
      std::max(4LL, ((long long)std::max(1, device_sm_count()) * kGatherWarpsPerSm + per_block - 1) / per_block);
  if (grid > cap_grid) grid = cap_grid;
  if (grid < 1) grid = 1;
  gather_kernel<<<(int)grid, kGatherThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      views, layer_lo, layer_hi, load_slot, load_pos, n_load, B, n_kv, cap, budget);
  return cudaGetLastError() == cudaSuccess ? SPC_OK : SPC_ERR_CUDA;
}

}  // namespace spc
