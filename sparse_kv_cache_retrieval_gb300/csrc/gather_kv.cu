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
// across the link, and a load of position p for KV head g reads the K and V
// rows of every layer of the launch as one contiguous run from one page. A
// work item is one 256-byte row (one load, one layer, K or V) copied by a
// half-warp; items are ordered (load, layer, K/V), so consecutive half-warps
// stream consecutive bytes of the host store, and spread over a grid-stride
// loop with 4 rows in flight per half-warp. The link saturates with about
// 0.5 MB in flight, which a small grid (one CTA of 512 threads per 8 SMs)
// already keeps: the rest of the GPU stays free for the kernels that run
// beside the gather on the other stream (attention, key scan). The flattened
// load index maps back to (request, KV head, i) through a prefix sum of
// n_load kept in shared memory.
#include "spc_device.cuh"
#include "spc_internal.h"

#include <algorithm>

namespace spc {

constexpr int kGatherThreads = 512;
#ifndef SPC_GATHER_UNROLL
#define SPC_GATHER_UNROLL 4
#endif
constexpr int kGatherUnroll = SPC_GATHER_UNROLL;
constexpr int kGatherMaxSeg = 1024;
#ifndef SPC_GATHER_SMS_PER_CTA
#define SPC_GATHER_SMS_PER_CTA 8
#endif
constexpr int kGatherSmsPerCta = SPC_GATHER_SMS_PER_CTA;   // one gather CTA per this many SMs

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
  const int NL = layer_hi - layer_lo;
  const int per_load = 2 * NL;                           // rows of one load: every layer, K and V
  const int total = R * per_load;                        // host limits keep this < 2^31
  const int l16 = tid & 15;
  const int hw0 = (blockIdx.x * kGatherThreads + tid) >> 4;
  const int nhw = (gridDim.x * kGatherThreads) >> 4;

  // Three stages per batch of kGatherUnroll rows of this half-warp: (A) locate
  // each row and load its (position, slot); (B) load the row from the host;
  // (C) store it to its slot. A runs one batch ahead of B, so the load of the
  // indices hides behind the previous batch's host round trip.
  int pos_n[kGatherUnroll], slot_n[kGatherUnroll];
  uint32_t hstride_n[kGatherUnroll];
  const uint16_t* hbase_n[kGatherUnroll];
  uint16_t* sbase_n[kGatherUnroll];
  auto stage_a = [&](int item0) {
#pragma unroll
    for (int u = 0; u < kGatherUnroll; ++u) {
      const int item = item0 + u * nhw;
      hbase_n[u] = nullptr;
      sbase_n[u] = nullptr;
      pos_n[u] = 0;
      slot_n[u] = 0;
      if (item >= total) continue;
      const int j = item / per_load;
      const int rem = item - j * per_load;
      const int layer = layer_lo + (rem >> 1);
      const int kv = rem & 1;
      // largest seg with pre[seg] <= j (segments with no load have equal bounds)
      int lo = 0, hi = nseg - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pre[mid] <= j) lo = mid; else hi = mid - 1;
      }
      const int seg = lo, i = j - pre[seg];
      const int b = seg / n_kv, g = seg - b * n_kv;
      const spc_gather_view vw = sv[b];
      const int lrel = layer - vw.layer0;
      const int lst = layer - vw.store_layer0;
      if (lrel < 0 || lrel >= vw.n_layers || lst < 0 || lst >= vw.store_layers) continue;
      const size_t li = (size_t)seg * K + i;
      pos_n[u] = load_pos[li];
      slot_n[u] = load_slot[li];
      // host row (p, g, lst, kv) = ((p * n_kv + g) * store_layers + lst) * 2 + kv
      hbase_n[u] = static_cast<const uint16_t*>(vw.host) +
                   (((size_t)g * vw.store_layers + lst) * 2 + kv) * kD + l16 * 8;
      sbase_n[u] = static_cast<uint16_t*>(vw.slots) + ((((size_t)lrel * 2 + kv) * n_kv + g) * K) * kD + l16 * 8;
      hstride_n[u] = (uint32_t)n_kv * (uint32_t)vw.store_layers * 2u * kD;   // elements per position
    }
  };

  stage_a(hw0);
  for (int item0 = hw0; item0 < total; item0 += nhw * kGatherUnroll) {
    uint4 v[kGatherUnroll];
    uint16_t* dst[kGatherUnroll];
#pragma unroll
    for (int u = 0; u < kGatherUnroll; ++u) {   // stage B of this batch
      dst[u] = nullptr;
      if (!hbase_n[u]) continue;
      v[u] = ldg_stream(hbase_n[u] + (size_t)pos_n[u] * hstride_n[u]);
      dst[u] = sbase_n[u] + (size_t)slot_n[u] * kD;
    }
    stage_a(item0 + nhw * kGatherUnroll);       // stage A of the next batch
#pragma unroll
    for (int u = 0; u < kGatherUnroll; ++u)     // stage C of this batch
      if (dst[u]) stg_v4(dst[u], v[u]);
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
  const long long max_items = (long long)(layer_hi - layer_lo) * 2 * B * n_kv * budget;
  const long long per_block = (kGatherThreads / 16) * kGatherUnroll;
  long long grid = (max_items + per_block - 1) / per_block;
  const long long cap_grid = std::max(4, device_sm_count() / kGatherSmsPerCta);
  if (grid > cap_grid) grid = cap_grid;
  if (grid < 1) grid = 1;
  gather_kernel<<<(int)grid, kGatherThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      views, layer_lo, layer_hi, load_slot, load_pos, n_load, B, n_kv, cap, budget);
  return cudaGetLastError() == cudaSuccess ? SPC_OK : SPC_ERR_CUDA;
}

}  // namespace spc
