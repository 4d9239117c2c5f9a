// Sparse GQA decode attention over the resident KV budget.
//
// Method: "ASPLOS'26 | SpeContext 让小模型先圈出重要 KV Cache" (marsggbo blog)
// §2 (softmax(QK^T/sqrt(d)) over the kept Top-K rows only) and §4 (the LLM
// forward runs on the sparse KV prepared in the previous iteration);
// "SpeContext: Enabling Efficient Long-context Reasoning with Speculative
// Context Sparsity in LLMs" (paperlayer.ai summary) §4.3 (for GQA the selected
// KV serves every query head of its group).
//
// GB300 design: the kept rows of one (layer, request, KV head) are split into
// chunks of 64 rows; a CTA walks a contiguous range of chunks with a 2-stage
// cp.async pipeline (16-byte copies; invalid rows are zero-filled), computes
// the G heads' base-2 scores with the lane-rotated half-warp reduce-scatter
// (one load of each K row serves the whole group), keeps an online softmax
// per head, and accumulates P.V with every thread owning (head, 8 columns)
// pairs so V rows are read once per row group. Split ranges are merged by the
// last CTA of the (layer, request, KV head), in split order (deterministic).
#include "spc_device.cuh"
#include "spc_internal.h"

namespace spc {

constexpr int kAttnThreads = 256;
constexpr int kAttnRows = 64;
constexpr int kAttnTargetCtas = 608;  // split so one launch fills the GPU ~4 CTAs deep
constexpr size_t kAttnStageBytes = (size_t)kAttnRows * kRowBytes;  // 16 KiB

template <int G>
struct AttnShape {
  static constexpr int HB = G < 8 ? G : 8;
  static constexpr int NHB = G / HB;
  static constexpr int PAIRS = G * 16;
  static constexpr int TPG = PAIRS < kAttnThreads ? PAIRS : kAttnThreads;
  static constexpr int RG = kAttnThreads / TPG;
  static constexpr int PPT = PAIRS / TPG;
};

struct AttnArgs {
  const uint16_t* q;
  const spc_kv_view* views;
  const int32_t* selected;
  const int32_t* slot_pos;
  float* out;
  float* part;
  uint32_t* counters;
  int B, n_q, n_kv, K, n_split, cps, n_chunks;
  float scale2;
};

template <int G>
__global__ void __launch_bounds__(kAttnThreads) attn_kernel(AttnArgs a) {
  using S = AttnShape<G>;
  extern __shared__ __align__(128) uint8_t asmem[];
  uint4* Ks = reinterpret_cast<uint4*>(asmem);                          // [2][64][16]
  uint4* Vs = reinterpret_cast<uint4*>(asmem + 2 * kAttnStageBytes);    // [2][64][16]
  float* q_s = reinterpret_cast<float*>(asmem + 4 * kAttnStageBytes);   // [G][128]
  float* sc = q_s + G * kD;                                             // [G][64]
  float* m_s = sc + G * kAttnRows;                                      // [G]
  float* l_s = m_s + G;                                                 // [G]
  float* al_s = l_s + G;                                                // [G]
  int* rowok = reinterpret_cast<int*>(al_s + G);                        // [2][64]
  __shared__ int s_last;

  const int split = blockIdx.x, g = blockIdx.y, lb = blockIdx.z;
  const int b = lb % a.B;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, l16 = lane & 15;
  const spc_kv_view vw = a.views[lb];
  const size_t seg = (size_t)b * a.n_kv + g;
  const int32_t* idx = (vw.use_slots ? a.slot_pos : a.selected) + seg * a.K;
  const uint16_t* kbase = static_cast<const uint16_t*>(vw.k) + (size_t)g * vw.rows * kD;
  const uint16_t* vbase = static_cast<const uint16_t*>(vw.v) + (size_t)g * vw.rows * kD;
  const int c0 = split * a.cps;
  const int c1 = min(c0 + a.cps, a.n_chunks);

  // q for the group, base-2 scaled
  const uint16_t* qg = a.q + ((size_t)lb * a.n_q + (size_t)g * G) * kD;
  for (int i = tid; i < G * kD; i += kAttnThreads)
    q_s[i] = __uint_as_float(uint32_t(qg[i]) << 16) * a.scale2;
  for (int h = tid; h < G; h += kAttnThreads) { m_s[h] = -INFINITY; l_s[h] = 0.f; }

  auto issue = [&](int c, int st) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int id = tid + k * kAttnThreads;
      const int r = id >> 5, part = id & 31, kv = part >> 4, ch = part & 15;
      const int i = c * kAttnRows + r;
      long long row = -1;
      if (i < a.K) {
        const int v = idx[i];
        if (v >= 0) row = vw.use_slots ? i : v;
        if (row >= vw.rows) row = -1;
      }
      const uint16_t* src = (kv ? vbase : kbase) + (size_t)(row < 0 ? 0 : row) * kD + ch * 8;
      uint4* dst = (kv ? Vs : Ks) + ((size_t)st * kAttnRows + r) * 16 + ch;
      cp_async16(dst, src, row < 0 ? 0 : 16);
      if (part == 0) rowok[st * kAttnRows + r] = row >= 0;
    }
  };

  // thread roles in P.V: (head, 8-column chunk) pairs, rows split over RG groups
  const int rg = tid / S::TPG, tp = tid - rg * S::TPG;
  const int cc = tp & 15, hbase = tp >> 4;
  float acc[S::PPT][8];
#pragma unroll
  for (int k = 0; k < S::PPT; ++k)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[k][e] = 0.f;

  float qr[S::HB][8];
  const int hw = tid >> 4;  // half-warp 0..15 -> rows [hw*4, hw*4+4)

  if (c0 < c1) {
    issue(c0, 0);
    cp_async_commit();
  }
  __syncthreads();  // q_s ready
  if (S::NHB == 1) {
#pragma unroll
    for (int h = 0; h < S::HB; ++h)
#pragma unroll
      for (int e = 0; e < 8; ++e) qr[h][e] = q_s[h * kD + l16 * 8 + e];
  }

  for (int c = c0; c < c1; ++c) {
    const int st = (c - c0) & 1;
    if (c + 1 < c1) {
      issue(c + 1, st ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();

    // ---- scores: 4 rows per half-warp, all heads of the group
    const uint4* kt = Ks + (size_t)st * kAttnRows * 16;
#pragma unroll 1
    for (int hb = 0; hb < S::NHB; ++hb) {
      if (S::NHB > 1) {
#pragma unroll
        for (int h = 0; h < S::HB; ++h)
#pragma unroll
          for (int e = 0; e < 8; ++e) qr[h][e] = q_s[(hb * S::HB + h) * kD + l16 * 8 + e];
      }
      float s4[4][S::HB];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 w = kt[(hw * 4 + (j ^ (l16 & 3))) * 16 + l16];
        float v[8];
        unpack8(w, v);
#pragma unroll
        for (int h = 0; h < S::HB; ++h) {
          float d0 = v[0] * qr[h][0];
#pragma unroll
          for (int e = 1; e < 8; ++e) d0 = fmaf(v[e], qr[h][e], d0);
          s4[j][h] = d0;
        }
      }
#pragma unroll
      for (int m = 2; m >= 1; m >>= 1)
#pragma unroll
        for (int j = 0; j < m; ++j)
#pragma unroll
          for (int h = 0; h < S::HB; ++h) s4[j][h] += __shfl_xor_sync(0xffffffffu, s4[j + m][h], m);
#pragma unroll
      for (int m = 4; m < 16; m <<= 1)
#pragma unroll
        for (int h = 0; h < S::HB; ++h) s4[0][h] += __shfl_xor_sync(0xffffffffu, s4[0][h], m);
      if (l16 < 4) {
        const int r = hw * 4 + l16;
        const bool ok = rowok[st * kAttnRows + r] != 0;
#pragma unroll
        for (int h = 0; h < S::HB; ++h) sc[(hb * S::HB + h) * kAttnRows + r] = ok ? s4[0][h] : -INFINITY;
      }
    }
    __syncthreads();

    // ---- online softmax per head (one warp per head)
    for (int h = warp; h < G; h += kAttnThreads / 32) {
      float* sh = sc + h * kAttnRows;
      const float x0 = sh[lane], x1 = sh[lane + 32];
      const float mo = m_s[h];
      const float mn = fmaxf(mo, warp_max(fmaxf(x0, x1)));
      const float p0 = mn == -INFINITY ? 0.f : exp2f(x0 - mn);
      const float p1 = mn == -INFINITY ? 0.f : exp2f(x1 - mn);
      sh[lane] = p0;
      sh[lane + 32] = p1;
      const float ps = warp_sum(p0 + p1);
      if (lane == 0) {
        const float alpha = (mn == -INFINITY) ? 1.f : exp2f(mo - mn);
        al_s[h] = alpha;
        l_s[h] = l_s[h] * alpha + ps;
        m_s[h] = mn;
      }
    }
    __syncthreads();

    // ---- P.V
    const uint4* vt = Vs + (size_t)st * kAttnRows * 16;
#pragma unroll
    for (int k = 0; k < S::PPT; ++k) {
      const float al = al_s[hbase + k * (S::TPG / 16)];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[k][e] *= al;
    }
    for (int r = rg; r < kAttnRows; r += S::RG) {
      const uint4 w = vt[r * 16 + cc];
      float v[8];
      unpack8(w, v);
#pragma unroll
      for (int k = 0; k < S::PPT; ++k) {
        const float p = sc[(hbase + k * (S::TPG / 16)) * kAttnRows + r];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[k][e] = fmaf(p, v[e], acc[k][e]);
      }
    }
    __syncthreads();
  }

  // ---- fold row groups, then write the output or this split's partial
  float* o_s = reinterpret_cast<float*>(asmem);  // [RG][G][128], reuses the K/V stages
#pragma unroll
  for (int k = 0; k < S::PPT; ++k) {
    float* dst = o_s + ((size_t)rg * G + hbase + k * (S::TPG / 16)) * kD + cc * 8;
#pragma unroll
    for (int e = 0; e < 8; ++e) dst[e] = acc[k][e];
  }
  __syncthreads();
  if (S::RG > 1) {
    for (int i = tid; i < G * kD; i += kAttnThreads) {
      float o = 0.f;
#pragma unroll
      for (int r = 0; r < S::RG; ++r) o += o_s[(size_t)r * G * kD + i];
      o_s[i] = o;  // row-group 0 slot; each i is owned by one thread
    }
    __syncthreads();
  }

  const size_t lbg = (size_t)lb * a.n_kv + g;
  float* outp = a.out + ((size_t)lb * a.n_q + (size_t)g * G) * kD;
  if (a.n_split == 1) {
    for (int i = tid; i < G * kD; i += kAttnThreads) {
      const float l = l_s[i / kD];
      outp[i] = l > 0.f ? o_s[i] / l : 0.f;
    }
    return;
  }
  float* pp = a.part + (lbg * a.n_split + split) * (size_t)G * (kD + 2);
  for (int i = tid; i < G * kD; i += kAttnThreads) pp[(i / kD) * (kD + 2) + 2 + (i % kD)] = o_s[i];
  for (int h = tid; h < G; h += kAttnThreads) {
    pp[h * (kD + 2)] = m_s[h];
    pp[h * (kD + 2) + 1] = l_s[h];
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(&a.counters[lbg], 1u) == (uint32_t)(a.n_split - 1));
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const float* pb = a.part + lbg * a.n_split * (size_t)G * (kD + 2);
  for (int i = tid; i < G * kD; i += kAttnThreads) {
    const int h = i / kD, c = i % kD;
    float M = -INFINITY;
    for (int s = 0; s < a.n_split; ++s) M = fmaxf(M, __ldcg(pb + ((size_t)s * G + h) * (kD + 2)));
    float Ls = 0.f, O = 0.f;
    if (M != -INFINITY) {
      for (int s = 0; s < a.n_split; ++s) {
        const float* ph = pb + ((size_t)s * G + h) * (kD + 2);
        const float ms = __ldcg(ph);
        const float w = ms == -INFINITY ? 0.f : exp2f(ms - M);
        Ls += __ldcg(ph + 1) * w;
        O += __ldcg(ph + 2 + c) * w;
      }
    }
    outp[i] = Ls > 0.f ? O / Ls : 0.f;
  }
  if (tid == 0) a.counters[lbg] = 0u;
}

static void attn_split(int n_layers, int B, int n_kv, int budget, int* n_split, int* cps,
                       int* n_chunks) {
  const int nc = (budget + kAttnRows - 1) / kAttnRows;
  const long long base = (long long)n_layers * B * n_kv;
  long long want = (kAttnTargetCtas + base - 1) / base;
  if (want < 1) want = 1;
  if (want > nc) want = nc;
  const int c = (int)((nc + want - 1) / want);
  *cps = c;
  *n_split = (nc + c - 1) / c;
  *n_chunks = nc;
}

template <int G>
static size_t attn_smem_bytes() {
  using S = AttnShape<G>;
  const size_t b = 4 * kAttnStageBytes +
                   sizeof(float) * ((size_t)G * kD + (size_t)G * kAttnRows + 3 * (size_t)G) +
                   sizeof(int) * 2 * kAttnRows;
  const size_t o = sizeof(float) * (size_t)S::RG * G * kD;
  return b > o ? b : o;
}

size_t attn_workspace(int n_layers, int B, int n_q, int n_kv, int budget) {
  int ns, cps, nc;
  attn_split(n_layers, B, n_kv, budget, &ns, &cps, &nc);
  const size_t nseg = (size_t)n_layers * B * n_kv;
  const size_t cnt = (nseg * sizeof(uint32_t) + 255) & ~size_t(255);
  const size_t part = ns > 1 ? nseg * ns * (size_t)(n_q / n_kv) * (kD + 2) * sizeof(float) : 0;
  return cnt + part;
}

template <int G>
static cudaError_t launch_attn(const AttnArgs& aa, dim3 grid, cudaStream_t st) {
  const size_t smem = attn_smem_bytes<G>();
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(attn_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  attn_kernel<G><<<grid, kAttnThreads, smem, st>>>(aa);
  return cudaGetLastError();
}

int attn_launch(const void* q, const spc_kv_view* views, const int32_t* selected,
                const int32_t* slot_pos, int n_layers, int B, int n_q, int n_kv, int budget,
                float scale, float* out, void* workspace, void* stream) {
  AttnArgs aa{};
  aa.q = static_cast<const uint16_t*>(q);
  aa.views = views;
  aa.selected = selected;
  aa.slot_pos = slot_pos;
  aa.out = out;
  const size_t nseg = (size_t)n_layers * B * n_kv;
  aa.counters = static_cast<uint32_t*>(workspace);
  aa.part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                     ((nseg * sizeof(uint32_t) + 255) & ~size_t(255)));
  aa.B = B; aa.n_q = n_q; aa.n_kv = n_kv; aa.K = budget;
  attn_split(n_layers, B, n_kv, budget, &aa.n_split, &aa.cps, &aa.n_chunks);
  aa.scale2 = scale * kLog2e;
  const dim3 grid(aa.n_split, n_kv, n_layers * B);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  switch (n_q / n_kv) {
    case 1: e = launch_attn<1>(aa, grid, st); break;
    case 2: e = launch_attn<2>(aa, grid, st); break;
    case 4: e = launch_attn<4>(aa, grid, st); break;
    case 8: e = launch_attn<8>(aa, grid, st); break;
    case 16: e = launch_attn<16>(aa, grid, st); break;
    case 32: e = launch_attn<32>(aa, grid, st); break;
    default: e = launch_attn<64>(aa, grid, st); break;
  }
  return e == cudaSuccess ? SPC_OK : SPC_ERR_CUDA;
}

}  // namespace spc

// ============================================================== no-allocation variant
// Scratch of spc_sparse_decode_attn_noalloc: a fixed area in the library's own
// device memory, so callers that cannot allocate device memory need not pass a
// workspace. Every device that loads the library holds these bytes until the
// process exits. Only host code needs its address (cudaGetSymbolAddress); the
// name itself is a host-side stand-in and must never be passed to a kernel.
#include <mutex>

namespace spc {

static __device__ __align__(256) unsigned char g_attn_noalloc_scratch[SPC_ATTN_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch area on the current device, looked up once
// per device (with that device current) and cached; nullptr on failure.
static void* attn_noalloc_scratch_address() {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_noalloc_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    addr[dev] = p;
  }
  return addr[dev];
}

int attn_noalloc_launch(const void* q, const spc_kv_view* views, const int32_t* selected,
                        const int32_t* slot_pos, int n_layers, int B, int n_q, int n_kv, int budget,
                        float scale, float* out, void* stream) {
  if (attn_workspace(n_layers, B, n_q, n_kv, budget) > SPC_ATTN_NOALLOC_SCRATCH_BYTES)
    return SPC_ERR_WORKSPACE;
  void* scratch = attn_noalloc_scratch_address();
  if (!scratch) return SPC_ERR_CUDA;
  // the split-merge counters must start at zero; the partials are always
  // written before they are read
  const size_t nseg = (size_t)n_layers * B * n_kv;
  if (cudaMemsetAsync(scratch, 0, nseg * sizeof(uint32_t), static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return SPC_ERR_CUDA;
  return attn_launch(q, views, selected, slot_pos, n_layers, B, n_q, n_kv, budget, scale, out,
                     scratch, stream);
}

}  // namespace spc
