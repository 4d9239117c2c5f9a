// C ABI entry points of libspc: argument validation on the host, then the
// launches. Every check runs before any CUDA call, so a rejected call touches
// neither the device nor the stream.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <map>
#include <mutex>
#include <tuple>

#include "spc.h"
#include "spc_device.cuh"
#include "spc_internal.h"

namespace spc {

constexpr int kMaxDevices = 64;

int device_sm_count() {
  static std::atomic<int> cached[kMaxDevices];   // 0 = not looked up yet
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 0 || dev >= kMaxDevices) {
    int n = 0;
    return cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess ? n : 0;
  }
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

bool tensor_map_bf16_sw128(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                           const uint64_t* strides, const uint32_t* box) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc || rank < 1 || rank > 5) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) st[i] = strides[i];
  }
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base), d, st, bx, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t set_func_attr(const void* fn, cudaFuncAttribute attr, int value) {
  // kernel attributes belong to a device's context: remember, per (kernel,
  // attribute, device), the largest value set so far
  static std::mutex mu;
  static std::map<std::tuple<const void*, int, int>, int> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_tuple(fn, (int)attr, dev);
  auto it = done.find(key);
  if (it != done.end() && it->second >= value) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, attr, value);
  if (e == cudaSuccess) done[key] = value;
  return e;
}

// ---------------------------------------------------------------- stream read
__global__ void __launch_bounds__(512) stream_read_kernel(const uint4* __restrict__ src, size_t n16,
                                                          uint32_t* sink) {
  uint32_t acc = 0;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n16; i += 4 * stride) {
    const uint4 a = ldg_stream(src + i), b = ldg_stream(src + i + stride);
    const uint4 c = ldg_stream(src + i + 2 * stride), d = ldg_stream(src + i + 3 * stride);
    acc ^= a.x ^ a.y ^ a.z ^ a.w ^ b.x ^ b.y ^ b.z ^ b.w ^ c.x ^ c.y ^ c.z ^ c.w ^ d.x ^ d.y ^ d.z ^ d.w;
  }
  for (; i < n16; i += stride) {
    const uint4 a = ldg_stream(src + i);
    acc ^= a.x ^ a.y ^ a.z ^ a.w;
  }
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, m);
  __shared__ uint32_t s[16];
  if ((threadIdx.x & 31) == 0) s[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t r = 0;
    for (int w = 0; w < 16; ++w) r ^= s[w];
    sink[blockIdx.x] = r;
  }
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Plain loads and stores (no read-only path): the host side of a mapped
// buffer may change between launches.
__global__ void __launch_bounds__(256) copy_kernel(uint8_t* __restrict__ dst, const uint8_t* __restrict__ src,
                                                   size_t bytes, int vec) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  const size_t t = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  size_t done = 0;
  if (vec) {
    const size_t n16 = bytes / 16;
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    size_t i = t;
    for (; i + 3 * stride < n16; i += 4 * stride) {
      const uint4 a = s4[i], b = s4[i + stride], c = s4[i + 2 * stride], d = s4[i + 3 * stride];
      d4[i] = a; d4[i + stride] = b; d4[i + 2 * stride] = c; d4[i + 3 * stride] = d;
    }
    for (; i < n16; i += stride) d4[i] = s4[i];
    done = n16 * 16;
  }
  for (size_t j = done + t; j < bytes; j += stride) dst[j] = src[j];
}

int copy_launch(void* dst, const void* src, size_t bytes, void* stream) {
  const bool vec = aligned16(dst) && aligned16(src);
  const size_t units = vec ? bytes / 16 : bytes;
  size_t grid = (units + 256 * 4 - 1) / (256 * 4);
  if (grid > 16) grid = 16;
  if (grid < 1) grid = 1;
  copy_kernel<<<(unsigned)grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint8_t*>(dst), static_cast<const uint8_t*>(src), bytes, vec ? 1 : 0);
  return cudaGetLastError() == cudaSuccess ? SPC_OK : SPC_ERR_CUDA;
}

int stream_read_launch(const void* src, size_t bytes, uint32_t* sink, int n_blocks, void* stream) {
  stream_read_kernel<<<n_blocks, 512, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(src), bytes / 16, sink);
  return cudaGetLastError() == cudaSuccess ? SPC_OK : SPC_ERR_CUDA;
}

static bool group_ok(int n_q, int n_kv) {
  if (n_q < 1 || n_kv < 1 || n_q % n_kv) return false;
  const int G = n_q / n_kv;
  return G == 1 || G == 2 || G == 4 || G == 8 || G == 16 || G == 32 || G == 64;
}

}  // namespace spc

using namespace spc;

extern "C" {

const char* spc_status_string(int status) {
  switch (status) {
    case SPC_OK: return "ok";
    case SPC_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer, bad flag)";
    case SPC_ERR_SHAPE: return "unsupported or inconsistent sizes";
    case SPC_ERR_CUDA: return "CUDA runtime or launch error";
    case SPC_ERR_TIMEOUT: return "a device-side wait timed out";
    case SPC_ERR_WORKSPACE: return "workspace missing or too small";
    case SPC_ERR_OVERFLOW: return "append would exceed the cache capacity";
    default: return "unknown status";
  }
}

int spc_version(void) { return 100; }

int spc_device_sm_count(void) { return device_sm_count(); }

size_t spc_score_select_workspace_size(int B, int H, int n_q, int n_kv, int d, int cap, int budget) {
  (void)budget;
  if (B < 1 || B > SPC_MAX_BATCH || H < 1 || d != SPC_HEAD_DIM || !group_ok(n_q, n_kv) || cap < 1)
    return 0;
  return score_select_workspace(B, H, n_q, n_kv, cap);
}

int spc_score_select_stages(const void* x, const void* Wq, const void* Wk, void* K_dlm, int32_t* len,
                            int append, int B, int H, int n_q, int n_kv, int d, int cap, int budget,
                            int n_sink, int n_recent, float* q_out, float* scores_out,
                            int32_t* selected, void* workspace, size_t workspace_bytes,
                            void* stream, int stages) {
  if (!x || !Wq || !K_dlm || !len || !selected) return SPC_ERR_INVALID_ARG;
  if (append != 0 && append != 1) return SPC_ERR_INVALID_ARG;
  if (stages < 1 || stages > 7) return SPC_ERR_INVALID_ARG;
  if (append && !Wk) return SPC_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(Wq) || (Wk && !aligned16(Wk)) || !aligned16(K_dlm) ||
      (q_out && !aligned16(q_out)))
    return SPC_ERR_INVALID_ARG;
  if (d != SPC_HEAD_DIM || !group_ok(n_q, n_kv)) return SPC_ERR_SHAPE;
  if (B < 1 || B > SPC_MAX_BATCH || H < 8 || H > SPC_MAX_HIDDEN || H % 8) return SPC_ERR_SHAPE;
  if (cap < 1 || cap > SPC_MAX_CAP) return SPC_ERR_SHAPE;
  if (budget < 1 || budget > SPC_MAX_BUDGET || budget > cap) return SPC_ERR_SHAPE;
  if (n_sink < 0 || n_recent < 0 || n_sink + n_recent > budget) return SPC_ERR_SHAPE;
  const size_t need = score_select_workspace(B, H, n_q, n_kv, cap);
  if (!workspace || workspace_bytes < need) return SPC_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return SPC_ERR_INVALID_ARG;
  ScoreSelectCall c{};
  c.x = x; c.Wq = Wq; c.Wk = Wk; c.K_dlm = K_dlm; c.len = len; c.append = append;
  c.B = B; c.H = H; c.n_q = n_q; c.n_kv = n_kv; c.cap = cap; c.budget = budget;
  c.n_sink = n_sink; c.n_recent = n_recent; c.q_out = q_out; c.scores_out = scores_out;
  c.selected = selected; c.workspace = workspace; c.stream = stream; c.stages = stages;
  return score_select_launch(c);
}

int spc_score_select(const void* x, const void* Wq, const void* Wk, void* K_dlm, int32_t* len,
                     int append, int B, int H, int n_q, int n_kv, int d, int cap, int budget,
                     int n_sink, int n_recent, float* q_out, float* scores_out,
                     int32_t* selected, void* workspace, size_t workspace_bytes, void* stream) {
  return spc_score_select_stages(x, Wq, Wk, K_dlm, len, append, B, H, n_q, n_kv, d, cap, budget,
                                 n_sink, n_recent, q_out, scores_out, selected, workspace,
                                 workspace_bytes, stream, SPC_STAGE_PROJECT | SPC_STAGE_SCAN | SPC_STAGE_SELECT);
}

int spc_elastic_diff(const int32_t* selected, const int32_t* slot_pos_prev, int32_t* slot_pos_next,
                     int32_t* load_slot, int32_t* load_pos, int32_t* n_load, int B, int n_kv,
                     int budget, int cap, void* stream) {
  if (!selected || !slot_pos_prev || !slot_pos_next || !load_slot || !load_pos || !n_load)
    return SPC_ERR_INVALID_ARG;
  if (B < 1 || n_kv < 1 || (long long)B * n_kv > 65535) return SPC_ERR_SHAPE;
  if (budget < 1 || budget > SPC_MAX_BUDGET || cap < 1 || cap > SPC_MAX_CAP) return SPC_ERR_SHAPE;
  return elastic_diff_launch(selected, slot_pos_prev, slot_pos_next, load_slot, load_pos, n_load, B,
                             n_kv, budget, cap, stream);
}

int spc_gather_kv(const spc_gather_view* views, int layer_lo, int layer_hi, const int32_t* load_slot,
                  const int32_t* load_pos, const int32_t* n_load, int B, int n_kv, int d, int cap,
                  int budget, void* stream) {
  if (!views || !load_slot || !load_pos || !n_load) return SPC_ERR_INVALID_ARG;
  if (d != SPC_HEAD_DIM) return SPC_ERR_SHAPE;
  if (B < 1 || B > SPC_MAX_BATCH || n_kv < 1 || B * n_kv > 1024) return SPC_ERR_SHAPE;
  if (layer_lo < 0 || layer_hi < layer_lo) return SPC_ERR_SHAPE;
  if (budget < 1 || budget > SPC_MAX_BUDGET || cap < 1 || cap > SPC_MAX_CAP) return SPC_ERR_SHAPE;
  if ((long long)(layer_hi - layer_lo) * 2 * B * n_kv * budget >= (1ll << 31)) return SPC_ERR_SHAPE;
  return gather_launch(views, layer_lo, layer_hi, load_slot, load_pos, n_load, B, n_kv, cap, budget,
                       stream);
}

size_t spc_sparse_decode_attn_workspace_size(int n_layers, int B, int n_q, int n_kv, int d, int budget) {
  if (n_layers < 1 || B < 1 || d != SPC_HEAD_DIM || !group_ok(n_q, n_kv) || budget < 1) return 0;
  return attn_workspace(n_layers, B, n_q, n_kv, budget);
}

int spc_fill_slots(const spc_gather_view* views, int layer_lo, int layer_hi, const int32_t* slot_pos,
                   int B, int n_kv, int d, int cap, int budget, void* stream) {
  if (!views || !slot_pos) return SPC_ERR_INVALID_ARG;
  if (d != SPC_HEAD_DIM) return SPC_ERR_SHAPE;
  if (B < 1 || B > SPC_MAX_BATCH || n_kv < 1 || B * n_kv > 1024) return SPC_ERR_SHAPE;
  if (layer_lo < 0 || layer_hi < layer_lo) return SPC_ERR_SHAPE;
  if (budget < 1 || budget > SPC_MAX_BUDGET || cap < 1 || cap > SPC_MAX_CAP) return SPC_ERR_SHAPE;
  return fill_slots_launch(views, layer_lo, layer_hi, slot_pos, B, n_kv, cap, budget, stream);
}

int spc_store_layer(void* store, const void* src, int n_kv, int d, int cap, int rows, int store_layers,
                    int layer, void* stream) {
  if (!store || !src) return SPC_ERR_INVALID_ARG;
  if (!aligned16(store) || !aligned16(src)) return SPC_ERR_INVALID_ARG;
  if (d != SPC_HEAD_DIM) return SPC_ERR_SHAPE;
  if (n_kv < 1 || n_kv > 1024 || cap < 1 || cap > SPC_MAX_CAP || rows < 0 || rows > cap) return SPC_ERR_SHAPE;
  if (store_layers < 1 || layer < 0 || layer >= store_layers) return SPC_ERR_SHAPE;
  return store_layer_launch(store, src, n_kv, cap, rows, store_layers, layer, stream);
}

int spc_offload_thresholds(int n_layers, int n_kv, int d, int B, int budget, int64_t kv_bytes,
                           int64_t* thresholds) {
  if (!thresholds) return SPC_ERR_INVALID_ARG;
  if (n_layers < 1 || n_kv < 1 || d < 1 || B < 1 || budget < 1 || kv_bytes < 0) return SPC_ERR_SHAPE;
  const long long row = 2LL * n_kv * d * 2;                       // K and V, every KV head, bf16
  const long long per_req_rows = kv_bytes / (row * B);            // rows one request may hold
  if (per_req_rows < (long long)n_layers * budget) return SPC_ERR_WORKSPACE;
  for (int k = 0; k < n_layers; ++k)
    thresholds[k] = (per_req_rows - (long long)k * budget) / (n_layers - k) + 1;
  thresholds[n_layers] = INT64_MAX;
  return SPC_OK;
}

int spc_sparse_decode_attn(const void* q, const spc_kv_view* views, const int32_t* selected,
                           const int32_t* slot_pos, int n_layers, int B, int n_q, int n_kv, int d,
                           int budget, float scale, float* out, void* workspace,
                           size_t workspace_bytes, void* stream) {
  if (!q || !views || !selected || !slot_pos || !out) return SPC_ERR_INVALID_ARG;
  if (d != SPC_HEAD_DIM || !group_ok(n_q, n_kv)) return SPC_ERR_SHAPE;
  if (n_layers < 1 || B < 1 || B > SPC_MAX_BATCH || (long long)n_layers * B > 65535) return SPC_ERR_SHAPE;
  if (n_kv > 65535 || budget < 1 || budget > SPC_MAX_BUDGET) return SPC_ERR_SHAPE;
  if (!(scale > 0.f)) return SPC_ERR_INVALID_ARG;
  const size_t need = attn_workspace(n_layers, B, n_q, n_kv, budget);
  if (!workspace || workspace_bytes < need) return SPC_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return SPC_ERR_INVALID_ARG;
  return attn_launch(q, views, selected, slot_pos, n_layers, B, n_q, n_kv, budget, scale, out,
                     workspace, stream);
}

int spc_sparse_decode_attn_noalloc(const void* q, const spc_kv_view* views, const int32_t* selected,
                                   const int32_t* slot_pos, int n_layers, int B, int n_q, int n_kv,
                                   int d, int budget, float scale, float* out, void* stream) {
  if (!q || !views || !selected || !slot_pos || !out) return SPC_ERR_INVALID_ARG;
  if (d != SPC_HEAD_DIM || !group_ok(n_q, n_kv)) return SPC_ERR_SHAPE;
  if (n_layers < 1 || B < 1 || B > SPC_MAX_BATCH || (long long)n_layers * B > 65535) return SPC_ERR_SHAPE;
  if (n_kv > 65535 || budget < 1 || budget > SPC_MAX_BUDGET) return SPC_ERR_SHAPE;
  if (!(scale > 0.f)) return SPC_ERR_INVALID_ARG;
  return attn_noalloc_launch(q, views, selected, slot_pos, n_layers, B, n_q, n_kv, budget, scale, out,
                             stream);
}

size_t spc_batch_select_workspace_size(int B, int cap, int budget) {
  if (B < 1 || B > SPC_MAX_BATCH || cap < 1 || cap > SPC_MAX_CAP || budget < 1 || budget > SPC_MAX_BUDGET) return 0;
  return batch_select_workspace(B, cap, budget);
}

int spc_batch_select(const float* scores, int32_t* len, int B, int n_kv, int cap, int budget, int n_sink,
                     int n_recent, int32_t* selected, void* workspace, size_t workspace_bytes, void* stream) {
  if (!scores || !len || !selected) return SPC_ERR_INVALID_ARG;
  if (B < 1 || B > SPC_MAX_BATCH || n_kv < 1 || n_kv > SPC_MAX_GROUP) return SPC_ERR_SHAPE;
  if (cap < 1 || cap > SPC_MAX_CAP) return SPC_ERR_SHAPE;
  if (budget < 1 || budget > SPC_MAX_BUDGET || budget > cap) return SPC_ERR_SHAPE;
  if (n_sink < 0 || n_recent < 0 || n_sink + n_recent > budget) return SPC_ERR_SHAPE;
  const size_t need = batch_select_workspace(B, cap, budget);
  if (!workspace || workspace_bytes < need) return SPC_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return SPC_ERR_INVALID_ARG;
  return batch_select_launch(scores, len, B, n_kv, cap, budget, n_sink, n_recent, selected, workspace, stream);
}

size_t spc_mla_score_select_workspace_size(int B, int H, int cap, int budget) {
  (void)budget;
  if (B < 1 || B > SPC_MAX_BATCH || H < 1 || cap < 1) return 0;
  return mla_score_select_workspace(B, cap);
}

int spc_mla_score_select(const void* x, const void* Wq, const void* Wuk, const void* Wdkv, void* C_dlm,
                         int32_t* len, int append, int B, int H, int cap, int budget, int n_sink,
                         int n_recent, float* scores_out, int32_t* selected, void* workspace,
                         size_t workspace_bytes, void* stream, int stages) {
  if (!x || !Wq || !Wuk || !C_dlm || !len || !selected) return SPC_ERR_INVALID_ARG;
  if (append != 0 && append != 1) return SPC_ERR_INVALID_ARG;
  if (stages < 1 || stages > 7) return SPC_ERR_INVALID_ARG;
  if (append && !Wdkv) return SPC_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(Wq) || !aligned16(Wuk) || (Wdkv && !aligned16(Wdkv)) || !aligned16(C_dlm))
    return SPC_ERR_INVALID_ARG;
  if (B < 1 || B > SPC_MAX_BATCH || H < 8 || H > SPC_MAX_HIDDEN || H % 8) return SPC_ERR_SHAPE;
  if (cap < 1 || cap > SPC_MAX_CAP) return SPC_ERR_SHAPE;
  if (budget < 1 || budget > SPC_MAX_BUDGET || budget > cap) return SPC_ERR_SHAPE;
  if (n_sink < 0 || n_recent < 0 || n_sink + n_recent > budget) return SPC_ERR_SHAPE;
  const size_t need = mla_score_select_workspace(B, cap);
  if (!workspace || workspace_bytes < need) return SPC_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return SPC_ERR_INVALID_ARG;
  MlaScoreSelectCall c{};
  c.x = x; c.Wq = Wq; c.Wuk = Wuk; c.Wdkv = Wdkv; c.C_dlm = C_dlm; c.len = len; c.append = append;
  c.B = B; c.H = H; c.cap = cap; c.budget = budget; c.n_sink = n_sink; c.n_recent = n_recent;
  c.scores_out = scores_out; c.selected = selected; c.workspace = workspace; c.stream = stream;
  c.stages = stages;
  return mla_score_select_launch(c);
}

int spc_mla_gather(const spc_gather_view* views, int layer_lo, int layer_hi, const int32_t* load_slot,
                   const int32_t* load_pos, const int32_t* n_load, int B, int cap, int budget,
                   void* stream) {
  if (!views || !load_slot || !load_pos || !n_load) return SPC_ERR_INVALID_ARG;
  if (B < 1 || B > SPC_MAX_BATCH) return SPC_ERR_SHAPE;
  if (layer_lo < 0 || layer_hi < layer_lo) return SPC_ERR_SHAPE;
  if (budget < 1 || budget > SPC_MAX_BUDGET || cap < 1 || cap > SPC_MAX_CAP) return SPC_ERR_SHAPE;
  return mla_gather_launch(views, layer_lo, layer_hi, load_slot, load_pos, n_load, B, budget, stream);
}

size_t spc_mla_decode_attn_workspace_size(int n_layers, int B, int budget) {
  if (n_layers < 1 || B < 1 || budget < 1 || budget > SPC_MAX_BUDGET) return 0;
  return mla_attn_workspace(n_layers, B, budget);
}

int spc_mla_decode_attn(const void* q, const void* Wuk, const void* Wuv, const spc_kv_view* views,
                        const int32_t* selected, const int32_t* slot_pos, int n_layers, int B, int budget,
                        float scale, float* out, void* workspace, size_t workspace_bytes, void* stream) {
  if (!q || !Wuk || !Wuv || !views || !selected || !slot_pos || !out) return SPC_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(Wuk) || !aligned16(Wuv) || !aligned16(out)) return SPC_ERR_INVALID_ARG;
  if (n_layers < 1 || B < 1 || B > SPC_MAX_BATCH || (long long)n_layers * B > 65535) return SPC_ERR_SHAPE;
  if (budget < 1 || budget > SPC_MAX_BUDGET) return SPC_ERR_SHAPE;
  if (!(scale > 0.f)) return SPC_ERR_INVALID_ARG;
  const size_t need = mla_attn_workspace(n_layers, B, budget);
  if (!workspace || workspace_bytes < need) return SPC_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return SPC_ERR_INVALID_ARG;
  return mla_attn_launch(q, Wuk, Wuv, views, selected, slot_pos, n_layers, B, budget, scale, out, workspace,
                         stream);
}

int spc_host_device_pointer(void* host_ptr, void** device_ptr) {
  if (!host_ptr || !device_ptr) return SPC_ERR_INVALID_ARG;
  void* p = nullptr;
  if (cudaHostGetDevicePointer(&p, host_ptr, 0) != cudaSuccess) {
    cudaGetLastError();
    return SPC_ERR_CUDA;
  }
  *device_ptr = p;
  return SPC_OK;
}

int spc_copy(void* dst, const void* src, size_t bytes, void* stream) {
  if (bytes == 0) return SPC_OK;
  if (!dst || !src) return SPC_ERR_INVALID_ARG;
  return copy_launch(dst, src, bytes, stream);
}

int spc_stream_read(const void* src, size_t bytes, uint32_t* sink, int n_blocks, void* stream) {
  if (!src || !sink || !aligned16(src)) return SPC_ERR_INVALID_ARG;
  if (bytes % 16 || n_blocks < 1 || n_blocks > 65535) return SPC_ERR_SHAPE;
  return stream_read_launch(src, bytes, sink, n_blocks, stream);
}

}  // extern "C"
