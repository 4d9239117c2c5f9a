// MLA variant of the decode hot path: query absorption, sparse attention over
// the selected latent rows, up-projection of its result, and the gather of
// missing latent rows from pinned host memory.
//
// Method: "ASPLOS'26 | SpeContext 让小模型先圈出重要 KV Cache" (marsggbo blog)
// §5: for DeepSeek's MLA the retrieval selects entries of the low-dimensional
// latent cache and only the selected entries are up-projected;
// "SpeContext: Enabling Efficient Long-context Reasoning with Speculative
// Context Sparsity in LLMs" (paperlayer.ai summary) §4.3: the retrieval stays
// head-level and only the selected latent entries are expanded for attention.
//
// A latent row is 576 bf16: a 512-value latent c shared by all heads and a
// 64-value decoupled rope key. Head h expands it into the key
// [W_uk[h] c ; c_rope] (192 values) and the value W_uv[h] c (128 values).
// Expanding each selected row and then attending is the same quantity as
//   score_h(r) = [W_uk[h]^T q_nope ; q_rope] . c_r        (query absorbed)
//   out_h      = W_uv[h] (sum_r softmax_r(score_h) c_r[:512])
// by associativity, so the up-projections are applied once per head (to the
// query, and to the softmax-weighted latent sum) instead of once per row; the
// rows themselves are only read, 1152 bytes each.
//
// GB300 design:
//  * mla_absorb_kernel: one CTA per (weight matrix, head) reads W_uk[h]
//    (128 x 512 bf16, 128 KiB) once and absorbs every query that uses it;
//  * mla_attn_kernel: per (layer, request) the kept rows are split into runs
//    of 32-row tiles, one CTA per run (two CTAs per SM). A producer warp copies
//    each tile's rows into a 2-stage ring with one bulk copy (cp.async.bulk)
//    per row, completion counted in bytes on the stage's mbarrier; rows sit
//    1168 bytes apart (16 bytes of padding) so ldmatrix is conflict-free, and
//    a 32-bit valid mask is published with the stage. Four consumer warps split S = Q C^T over the
//    576 dims (9 k-steps of mma.sync m16n8k16 each; the 16 heads are the M
//    side, the absorbed query rounded to bf16), sum the four partial S tiles
//    through shared memory, run the online softmax in base 2, and compute
//    O += P C[:, :512]
//    with each warp owning 128 of the 512 latent dims (P in bf16 high + low
//    parts from shared memory, the rows as ldmatrix.trans B fragments). Each
//    CTA writes its (max, sum, O) partial to the workspace;
//  * mla_out_kernel: per (layer, request, head, 32 output values) merges the
//    partials in a fixed order (deterministic) and applies those 32 rows of
//    W_uv[h] (128 x 512 bf16).
//  * mla_gather_kernel: one warp per load streams the load's run of the
//    position-major host store (every stored layer's latent row of that
//    position, contiguous) into the layer slots.
#include <cuda_bf16.h>

#include <algorithm>

#include "spc_device.cuh"
#include "spc_internal.h"

namespace spc {

constexpr int kLat = SPC_MLA_LATENT + SPC_MLA_ROPE;   // 576 values per latent row
constexpr int kLatBytes = kLat * 2;                   // 1152
constexpr int kLatPieces = kLatBytes / 16;            // 72 16-byte pieces
constexpr int kDc = SPC_MLA_LATENT;                   // 512
constexpr int kNope = SPC_MLA_NOPE;                   // 128
constexpr int kDv = SPC_MLA_V;                        // 128
constexpr int kQk = SPC_MLA_NOPE + SPC_MLA_ROPE;      // 192
constexpr int kMH = SPC_MLA_HEADS;                    // 16
constexpr long long kMlaWait = 4000000000ll;          // bounded mbarrier waits (clock cycles, ~2 s)

// ============================================================== absorption
constexpr int kAbsThreads = 256;   // 16 row groups x 16 lanes of 8 latent coordinates
constexpr int kAbsRg = 16;
constexpr int kAbsChunk = 128;     // latent coordinates per CTA (4 CTAs per head)

template <typename QT>
__device__ __forceinline__ float load_q(const QT* p);
template <>
__device__ __forceinline__ float load_q<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float load_q<uint16_t>(const uint16_t* p) { return __uint_as_float(uint32_t(*p) << 16); }

// qa[i, h] = [W_uk[w(i), h]^T q[i, h, :128] ; q[i, h, 128:192]] for items i
// of weight matrix w(i) = i / items_per_w. Grid (heads, weight matrices,
// 4 coordinate chunks x item chunks of NI): a CTA reads a 128-coordinate
// column block of W_uk[w, h] (32 KiB, 16-byte loads, 8 rows in flight per
// thread), each of 16 row groups sums 8 of the 128 nope rows, and the row
// groups are added through shared memory.
template <typename QT, int NI>
__global__ void __launch_bounds__(kAbsThreads)
mla_absorb_kernel(const QT* __restrict__ q, const uint16_t* __restrict__ Wuk, int n_items, int items_per_w,
                  float* __restrict__ qa) {
  __shared__ float qs[kNope][NI];
  __shared__ __align__(16) float red[kAbsRg * NI * kAbsChunk];
  const int h = blockIdx.x, w = blockIdx.y, chunk = blockIdx.z & 3, zi = blockIdx.z >> 2, tid = threadIdx.x;
  const int i0 = w * items_per_w + zi * NI;
  const int i1 = min(min(n_items, (w + 1) * items_per_w), i0 + NI);
  const int ni = i1 - i0;
  if (ni <= 0) return;
  const int rg = tid >> 4, cl = tid & 15;
  // W_uk[w, h] is [128][512]: row j holds the weights of nope value j; this
  // thread's 8 rows are requested before the queries are staged
  const uint16_t* W = Wuk + ((size_t)w * kMH + h) * kNope * kDc + chunk * kAbsChunk + cl * 8;
  uint4 wv[kNope / kAbsRg];
#pragma unroll
  for (int k = 0; k < kNope / kAbsRg; ++k) wv[k] = ldg_stream(W + (size_t)(rg + kAbsRg * k) * kDc);
  for (int idx = tid; idx < kNope * NI; idx += kAbsThreads) {
    const int j = idx / NI, it = idx - j * NI;
    qs[j][it] = it < ni ? load_q<QT>(q + ((size_t)(i0 + it) * kMH + h) * kQk + j) : 0.f;
  }
  if (chunk == 0) {
    for (int idx = tid; idx < ni * SPC_MLA_ROPE; idx += kAbsThreads) {
      const int it = idx / SPC_MLA_ROPE, k = idx - it * SPC_MLA_ROPE;
      qa[((size_t)(i0 + it) * kMH + h) * kLat + kDc + k] =
          load_q<QT>(q + ((size_t)(i0 + it) * kMH + h) * kQk + kNope + k);
    }
  }
  __syncthreads();
  float acc[NI][8];
#pragma unroll
  for (int it = 0; it < NI; ++it)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[it][e] = 0.f;
#pragma unroll
  for (int k = 0; k < kNope / kAbsRg; ++k) {
    float f[8];
    unpack8(wv[k], f);
    const int j = rg + kAbsRg * k;
#pragma unroll
    for (int it = 0; it < NI; ++it) {
      const float qv = qs[j][it];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[it][e] = fmaf(f[e], qv, acc[it][e]);
    }
  }
#pragma unroll
  for (int it = 0; it < NI; ++it) {
    float4* dst = reinterpret_cast<float4*>(red + ((size_t)(rg * NI + it) * kAbsChunk + cl * 8));
    dst[0] = make_float4(acc[it][0], acc[it][1], acc[it][2], acc[it][3]);
    dst[1] = make_float4(acc[it][4], acc[it][5], acc[it][6], acc[it][7]);
  }
  __syncthreads();
  for (int o = tid; o < ni * kAbsChunk; o += kAbsThreads) {
    const int it = o / kAbsChunk, c = o - it * kAbsChunk;
    float sum = 0.f;
#pragma unroll
    for (int g = 0; g < kAbsRg; ++g) sum += red[(g * NI + it) * kAbsChunk + c];
    qa[((size_t)(i0 + it) * kMH + h) * kLat + chunk * kAbsChunk + c] = sum;
  }
}

template <typename QT>
static void absorb_launch_t(const QT* q, const uint16_t* Wuk, int n_items, int items_per_w, float* qa,
                            cudaStream_t st) {
  const int n_w = (n_items + items_per_w - 1) / items_per_w;
  const int ni = items_per_w <= 1 ? 1 : items_per_w <= 2 ? 2 : 4;
  const dim3 grid(kMH, n_w, 4 * ((items_per_w + ni - 1) / ni));
  if (ni == 1) mla_absorb_kernel<QT, 1><<<grid, kAbsThreads, 0, st>>>(q, Wuk, n_items, items_per_w, qa);
  else if (ni == 2) mla_absorb_kernel<QT, 2><<<grid, kAbsThreads, 0, st>>>(q, Wuk, n_items, items_per_w, qa);
  else mla_absorb_kernel<QT, 4><<<grid, kAbsThreads, 0, st>>>(q, Wuk, n_items, items_per_w, qa);
}

int mla_absorb_launch(const void* q, int q_bf16, const void* Wuk, int n_items, int items_per_w, float* qa,
                      void* stream) {
  if (n_items <= 0) return SPC_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (q_bf16)
    absorb_launch_t(static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(Wuk), n_items, items_per_w, qa, st);
  else
    absorb_launch_t(static_cast<const float*>(q), static_cast<const uint16_t*>(Wuk), n_items, items_per_w, qa, st);
  return cudaGetLastError() == cudaSuccess ? SPC_OK : SPC_ERR_CUDA;
}

// ============================================================== attention
constexpr int kMaRows = 32;                          // latent rows per tile
constexpr int kMaStages = 2;
constexpr int kMaCWarps = 4;
constexpr int kMaCThreads = kMaCWarps * 32;
constexpr int kMaThreads = kMaCThreads + 32;         // + producer warp
constexpr int kMaPitch = kLatBytes + 16;             // 1168: rows 16 bytes apart in bank groups, so
                                                     // ldmatrix over 8 rows is conflict-free
constexpr uint32_t kMaTile = kMaRows * kMaPitch;     // 36.5 KiB
constexpr int kMaKs = kLat / 16 / kMaCWarps;         // 9 k-steps of S per warp
constexpr int kMaPStride = 40;                       // bf16 per P row (32 + 8: conflict-free ldmatrix)
constexpr int kMaTargetCtas = 304;                   // two CTAs per SM of a 152-SM GB300
constexpr int kMaPart = kDc + 4;                     // partial record: m, l, pad, pad, o[512]

struct MaSmem {
  static constexpr size_t stages = (size_t)kMaStages * kMaTile;
  static constexpr size_t red = (size_t)kMaCWarps * 4 * 32 * 16;     // S partials [warp][ntile][lane] float4
  static constexpr size_t p = 2 * kMH * kMaPStride * 2;              // P high and low, bf16
  static constexpr size_t mx = kMaCWarps * kMH * 4;                  // per-warp tile maxima
  static constexpr size_t ls = kMaCWarps * kMH * 4;                  // per-warp sums
  static constexpr size_t bars = 8 * 3 * kMaStages;                  // valid masks, full, empty
  static constexpr size_t total = stages + red + p + mx + ls + bars;
};

struct MlaAttnArgs {
  const float* qa;               // [units][16][576] absorbed queries (unscaled)
  const spc_kv_view* views;      // [units]: k = latent rows [rows][576]
  const int32_t* selected;       // [B][budget]
  const int32_t* slot_pos;       // [B][budget]
  float* part;                   // [units][n_split][16][kMaPart]
  int* status;
  int B, K, n_split, tpc;
  float scale2;                  // scale * log2(e)
};

__device__ __forceinline__ void ma_bar() { asm volatile("bar.sync 1, %0;" :: "n"(kMaCThreads) : "memory"); }

// two CTAs per SM: ten warps over four sub-partitions of 16K registers leave
// 168 registers per thread
__global__ void __launch_bounds__(kMaThreads, 2) mla_attn_kernel(MlaAttnArgs a) {
  extern __shared__ __align__(128) uint8_t msm[];
  float4* red = reinterpret_cast<float4*>(msm + MaSmem::stages);
  uint16_t* pbuf = reinterpret_cast<uint16_t*>(msm + MaSmem::stages + MaSmem::red);       // [2][16][40]
  float* mxs = reinterpret_cast<float*>(msm + MaSmem::stages + MaSmem::red + MaSmem::p);   // [4][16]
  float* lss = mxs + kMaCWarps * kMH;                                                      // [4][16]
  uint64_t* vmask = reinterpret_cast<uint64_t*>(lss + kMaCWarps * kMH);
  uint64_t* full = vmask + kMaStages;
  uint64_t* empty = full + kMaStages;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int unit = blockIdx.x / a.n_split, split = blockIdx.x - unit * a.n_split;
  const int b = unit % a.B;
  const int n_tiles = (a.K + kMaRows - 1) / kMaRows;
  const int t0 = min(n_tiles, split * a.tpc), t1 = min(n_tiles, t0 + a.tpc);

  if (tid == 0) {
    for (int s = 0; s < kMaStages; ++s) {
      mbar_init(&full[s], 1);        // lane 0: mask published, 32 row copies expected
      mbar_init(&empty[s], kMaCWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kMaCWarps) {
    // ================= producer: lane r resolves row r of each tile
    const spc_kv_view vw = a.views[unit];
    const uint16_t* base = static_cast<const uint16_t*>(vw.k);
    const int32_t* sel = a.selected + (size_t)b * a.K;
    const int32_t* spos = a.slot_pos + (size_t)b * a.K;
    int it = 0;
    for (int t = t0; t < t1; ++t, ++it) {
      const int s = it % kMaStages;
      const uint32_t ph = (it / kMaStages) & 1;
      const int i = t * kMaRows + lane;
      int r = -1;
      if (i < a.K) {
        if (vw.use_slots) r = spos[i] >= 0 ? i : -1;
        else r = sel[i];
      }
      if (r >= vw.rows) r = -1;
      const uint32_t ok = __ballot_sync(0xffffffffu, r >= 0);
      if (!mbar_wait_bounded(&empty[s], ph ^ 1, kMlaWait)) {
        if (lane == 0) set_status(a.status, SPC_ERR_TIMEOUT);
        break;
      }
      // one bulk copy per row, lane r copying row r of the tile; a row not
      // kept copies the view's row 0 instead (finite values: its logits are
      // masked, so its weight is exactly 0)
      if (lane == 0) {
        vmask[s] = ok;
        mbar_arrive_expect_tx(&full[s], kMaRows * kLatBytes);
      }
      __syncwarp();
      bulk_g2s(msm + (size_t)s * kMaTile + lane * kMaPitch, base + (size_t)(r < 0 ? 0 : r) * kLat, kLatBytes,
               &full[s]);
    }
    for (int k = max(0, it - kMaStages); k < it; ++k)
      mbar_wait_bounded(&full[k % kMaStages], (k / kMaStages) & 1, kMlaWait);
    __syncwarp();
    return;
  }

  // ================= consumers
  const int kw = warp;                                // k-split slice of S, 128-dim slice of O
  const int gid = lane >> 2, tig = lane & 3, lm = lane >> 3, lr = lane & 7;
  const uint32_t smem0 = smem_u32(msm);
  const uint32_t pb0 = smem_u32(pbuf);
  bool dead = false;

  // absorbed query fragments of this warp's 9 k-steps, rounded to bf16 (the
  // scores carry the query's 2^-9 relative rounding; P keeps ~16 bits below)
  const float* qp = a.qa + (size_t)unit * kMH * kLat;
  uint32_t qh[kMaKs][4];
#pragma unroll
  for (int ks = 0; ks < kMaKs; ++ks) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int h = gid + ((e & 1) ? 8 : 0);
      const int c = (kw * kMaKs + ks) * 16 + tig * 2 + ((e & 2) ? 8 : 0);
      const float2 v = *reinterpret_cast<const float2*>(qp + (size_t)h * kLat + c);
      qh[ks][e] = pack_bf16(v.x * a.scale2, v.y * a.scale2);
    }
  }
  float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
  float o[16][4];
#pragma unroll
  for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

  int it = 0;
  for (int t = t0; t < t1; ++t, ++it) {
    const int s = it % kMaStages;
    const uint32_t ph = (it / kMaStages) & 1;
    if (!dead && !mbar_wait_bounded(&full[s], ph, kMlaWait)) {
      if (lane == 0) set_status(a.status, SPC_ERR_TIMEOUT);
      dead = true;
    }
    const uint32_t okm = dead ? 0u : (uint32_t)vmask[s];
    const uint32_t tb = smem0 + (uint32_t)(s * kMaTile);

    // ---- partial S over this warp's 144 dims: 16 heads x 32 rows
    float acc[4][4];
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[n][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < kMaKs; ++ks) {
      const int kg = kw * kMaKs + ks;
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        const int row = np * 16 + ((lm >> 1) << 3) + lr;
        uint32_t b0, b1, b2, b3;
        ldsm_x4(tb + row * kMaPitch + ((kg * 2 + (lm & 1)) << 4), b0, b1, b2, b3);
        mma_bf16(acc[2 * np], qh[ks], b0, b1);
        mma_bf16(acc[2 * np + 1], qh[ks], b2, b3);
      }
    }
#pragma unroll
    for (int n = 0; n < 4; ++n) red[(kw * 4 + n) * 32 + lane] = make_float4(acc[n][0], acc[n][1], acc[n][2], acc[n][3]);
    ma_bar();
    // ---- this warp finishes rows kw*8 .. kw*8+7 (n-tile kw): heads gid (x, y)
    // and gid + 8 (z, w) at rows kw*8 + 2 tig, +1
    float4 v = red[(0 * 4 + kw) * 32 + lane];
#pragma unroll
    for (int w = 1; w < kMaCWarps; ++w) {
      const float4 u = red[(w * 4 + kw) * 32 + lane];
      v.x += u.x; v.y += u.y; v.z += u.z; v.w += u.w;
    }
    const int r0 = kw * 8 + tig * 2;
    const bool v0 = (okm >> r0) & 1u, v1 = (okm >> (r0 + 1)) & 1u;
    if (!v0) v.x = v.z = -INFINITY;
    if (!v1) v.y = v.w = -INFINITY;
    float tm_lo = fmaxf(v.x, v.y), tm_hi = fmaxf(v.z, v.w);
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
      tm_lo = fmaxf(tm_lo, __shfl_xor_sync(0xffffffffu, tm_lo, off));
      tm_hi = fmaxf(tm_hi, __shfl_xor_sync(0xffffffffu, tm_hi, off));
    }
    if (tig == 0) {
      mxs[kw * kMH + gid] = tm_lo;
      mxs[kw * kMH + gid + 8] = tm_hi;
    }
    ma_bar();
    float mx_lo = mxs[gid], mx_hi = mxs[gid + 8];
#pragma unroll
    for (int w = 1; w < kMaCWarps; ++w) {
      mx_lo = fmaxf(mx_lo, mxs[w * kMH + gid]);
      mx_hi = fmaxf(mx_hi, mxs[w * kMH + gid + 8]);
    }
    const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
    const float al_lo = mn_lo == -INFINITY ? 1.f : exp2f(m_lo - mn_lo);
    const float al_hi = mn_hi == -INFINITY ? 1.f : exp2f(m_hi - mn_hi);
    const float p0 = mn_lo == -INFINITY ? 0.f : exp2f(v.x - mn_lo);
    const float p1 = mn_lo == -INFINITY ? 0.f : exp2f(v.y - mn_lo);
    const float p2 = mn_hi == -INFINITY ? 0.f : exp2f(v.z - mn_hi);
    const float p3 = mn_hi == -INFINITY ? 0.f : exp2f(v.w - mn_hi);
    // this warp's share of the row sums (its 8 rows); the warps' shares are
    // added at the end, all rescaled by the same factors
    float sl = p0 + p1, sh = p2 + p3;
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
      sl += __shfl_xor_sync(0xffffffffu, sl, off);
      sh += __shfl_xor_sync(0xffffffffu, sh, off);
    }
    l_lo = l_lo * al_lo + sl;
    l_hi = l_hi * al_hi + sh;
    m_lo = mn_lo;
    m_hi = mn_hi;
    {
      const float h0 = bf16_round(p0), h1 = bf16_round(p1), h2 = bf16_round(p2), h3 = bf16_round(p3);
      uint32_t* ph32 = reinterpret_cast<uint32_t*>(pbuf);
      uint32_t* pl32 = reinterpret_cast<uint32_t*>(pbuf + kMH * kMaPStride);
      ph32[(gid * kMaPStride + r0) / 2] = pack_bf16(h0, h1);
      ph32[((gid + 8) * kMaPStride + r0) / 2] = pack_bf16(h2, h3);
      pl32[(gid * kMaPStride + r0) / 2] = pack_bf16(p0 - h0, p1 - h1);
      pl32[((gid + 8) * kMaPStride + r0) / 2] = pack_bf16(p2 - h2, p3 - h3);
    }
    ma_bar();
    // ---- O (16 heads x this warp's 128 latent dims) += P C[:, kw*128 ..]
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      o[n][0] *= al_lo; o[n][1] *= al_lo;
      o[n][2] *= al_hi; o[n][3] *= al_hi;
    }
#pragma unroll
    for (int kk = 0; kk < kMaRows / 16; ++kk) {
      uint32_t ah[4], alw[4];
      const uint32_t pa = pb0 + (uint32_t)((((lm & 1) << 3) + lr) * kMaPStride + kk * 16 + ((lm >> 1) << 3)) * 2;
      ldsm_x4(pa, ah[0], ah[1], ah[2], ah[3]);
      ldsm_x4(pa + kMH * kMaPStride * 2, alw[0], alw[1], alw[2], alw[3]);
      const int row = kk * 16 + ((lm & 1) << 3) + lr;
#pragma unroll
      for (int np = 0; np < 8; ++np) {
        const int piece = kw * 16 + np * 2 + (lm >> 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(tb + row * kMaPitch + (piece << 4), b0, b1, b2, b3);
        mma_bf16(o[2 * np], ah, b0, b1);
        mma_bf16(o[2 * np], alw, b0, b1);
        mma_bf16(o[2 * np + 1], ah, b2, b3);
        mma_bf16(o[2 * np + 1], alw, b2, b3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }

  // ---- this CTA's partial: m per head (equal in every warp), l summed over
  // the warps, O of this warp's 128 dims
  if (tig == 0) {
    lss[kw * kMH + gid] = l_lo;
    lss[kw * kMH + gid + 8] = l_hi;
  }
  ma_bar();
  float* pr = a.part + ((size_t)unit * a.n_split + split) * kMH * kMaPart;
  if (kw == 0 && tig == 0) {
    float s_lo = 0.f, s_hi = 0.f;
#pragma unroll
    for (int w = 0; w < kMaCWarps; ++w) { s_lo += lss[w * kMH + gid]; s_hi += lss[w * kMH + gid + 8]; }
    *reinterpret_cast<float2*>(pr + (size_t)gid * kMaPart) = make_float2(m_lo, s_lo);
    *reinterpret_cast<float2*>(pr + (size_t)(gid + 8) * kMaPart) = make_float2(m_hi, s_hi);
  }
#pragma unroll
  for (int n = 0; n < 16; ++n) {
    const int c = kw * 128 + n * 8 + tig * 2;
    *reinterpret_cast<float2*>(pr + (size_t)gid * kMaPart + 4 + c) = make_float2(o[n][0], o[n][1]);
    *reinterpret_cast<float2*>(pr + (size_t)(gid + 8) * kMaPart + 4 + c) = make_float2(o[n][2], o[n][3]);
  }
}

// ============================================================== merge + W_uv
constexpr int kMoThreads = 256;
constexpr int kMoChunk = 32;       // output values per CTA (4 CTAs per head)

// Grid (units, heads, 4 chunks of 32 output values): merge the head's split
// partials in a fixed order (every CTA of the head the same way), then 8 warps
// x 4 values each dot W_uv[l, h][v, :] with the merged latent sum, two
// 16-byte loads per value and lane, all 8 in flight.
__global__ void __launch_bounds__(kMoThreads)
mla_out_kernel(const float* __restrict__ part, const uint16_t* __restrict__ Wuv, int B, int n_split,
               float* __restrict__ out) {
  __shared__ __align__(16) float lat[kDc];
  __shared__ float wgt[64];
  const int unit = blockIdx.x, h = blockIdx.y, v0 = blockIdx.z * kMoChunk, tid = threadIdx.x;
  const int l = unit / B;
  const int warp = tid >> 5, lane = tid & 31;
  // this warp's 4 rows of W_uv[l, h] are requested first: they do not depend
  // on the merge, so their DRAM latency overlaps it
  const uint16_t* W = Wuv + ((size_t)l * kMH + h) * kDv * kDc;
  const int vb = v0 + warp * 4;
  uint4 w0[4], w1[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    w0[u] = ldg_stream(W + (size_t)(vb + u) * kDc + lane * 8);
    w1[u] = ldg_stream(W + (size_t)(vb + u) * kDc + 256 + lane * 8);
  }
  const float* pp = part + (size_t)unit * n_split * kMH * kMaPart + (size_t)h * kMaPart;
  const size_t sstride = (size_t)kMH * kMaPart;
  // split weights exp2(m_s - M) / sum_s exp2(m_s - M) l_s, by warp 0 (two
  // splits per lane, all loads in flight together; n_split <= 64)
  if (tid < 32) {
    const bool h0 = tid < n_split, h1 = tid + 32 < n_split;
    const float2 a0 = h0 ? *reinterpret_cast<const float2*>(pp + tid * sstride) : make_float2(-INFINITY, 0.f);
    const float2 a1 = h1 ? *reinterpret_cast<const float2*>(pp + (tid + 32) * sstride) : make_float2(-INFINITY, 0.f);
    const float M = warp_max(fmaxf(a0.x, a1.x));
    const float e0 = M == -INFINITY || !h0 ? 0.f : exp2f(a0.x - M);
    const float e1 = M == -INFINITY || !h1 ? 0.f : exp2f(a1.x - M);
    const float den = warp_sum(e0 * a0.y + e1 * a1.y);
    const float inv = den > 0.f ? 1.f / den : 0.f;
    if (h0) wgt[tid] = e0 * inv;
    if (h1) wgt[tid + 32] = e1 * inv;
  }
  __syncthreads();
  if (tid < kDc / 4) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < n_split; ++s) {
      const float w = wgt[s];
      const float4 v = *reinterpret_cast<const float4*>(pp + s * sstride + 4 + 4 * tid);
      acc.x = fmaf(w, v.x, acc.x); acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z); acc.w = fmaf(w, v.w, acc.w);
    }
    *reinterpret_cast<float4*>(lat + 4 * tid) = acc;
  }
  __syncthreads();
  float lv[16];
#pragma unroll
  for (int e = 0; e < 8; ++e) { lv[e] = lat[lane * 8 + e]; lv[8 + e] = lat[256 + lane * 8 + e]; }
  float sum[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    float f0[8], f1[8];
    unpack8(w0[u], f0);
    unpack8(w1[u], f1);
    float sacc = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) sacc = fmaf(f0[e], lv[e], fmaf(f1[e], lv[8 + e], sacc));
    sum[u] = warp_sum(sacc);
  }
  const float r = lane == 0 ? sum[0] : lane == 1 ? sum[1] : lane == 2 ? sum[2] : sum[3];
  if (lane < 4) out[((size_t)unit * kMH + h) * kDv + vb + lane] = r;
}

static void mla_attn_plan(int units, int budget, int* n_split, int* tpc) {
  const int n_tiles = (budget + kMaRows - 1) / kMaRows;
  int s = (kMaTargetCtas + units - 1) / units;
  s = std::max(1, std::min(s, std::min(n_tiles, 64)));
  const int t = (n_tiles + s - 1) / s;
  *tpc = t;
  *n_split = (n_tiles + t - 1) / t;
}

static size_t mla_part_bytes(int units, int budget) {
  int ns, tpc;
  mla_attn_plan(units, budget, &ns, &tpc);
  return (((size_t)units * ns * kMH * kMaPart * sizeof(float)) + 255) & ~size_t(255);
}

size_t mla_attn_workspace(int n_layers, int B, int budget) {
  const int units = n_layers * B;
  const size_t qa = (((size_t)units * kMH * kLat * sizeof(float)) + 255) & ~size_t(255);
  return 256 + qa + mla_part_bytes(units, budget);
}

int mla_attn_launch(const void* q, const void* Wuk, const void* Wuv, const spc_kv_view* views,
                    const int32_t* selected, const int32_t* slot_pos, int n_layers, int B, int budget,
                    float scale, float* out, void* workspace, void* stream) {
  const int units = n_layers * B;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* status = reinterpret_cast<int*>(ws);
  float* qa = reinterpret_cast<float*>(ws + 256);
  float* part = reinterpret_cast<float*>(ws + 256 + ((((size_t)units * kMH * kLat * sizeof(float)) + 255) & ~size_t(255)));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int rc = mla_absorb_launch(q, 1, Wuk, units, B, qa, stream);
  if (rc != SPC_OK) return rc;
  MlaAttnArgs aa{};
  aa.qa = qa; aa.views = views; aa.selected = selected; aa.slot_pos = slot_pos; aa.part = part;
  aa.status = status; aa.B = B; aa.K = budget;
  mla_attn_plan(units, budget, &aa.n_split, &aa.tpc);
  aa.scale2 = scale * kLog2e;
  if (set_func_attr((const void*)mla_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                    (int)MaSmem::total) != cudaSuccess)
    return SPC_ERR_CUDA;
  mla_attn_kernel<<<units * aa.n_split, kMaThreads, MaSmem::total, st>>>(aa);
  if (cudaGetLastError() != cudaSuccess) return SPC_ERR_CUDA;
  mla_out_kernel<<<dim3(units, kMH, kDv / kMoChunk), kMoThreads, 0, st>>>(part, static_cast<const uint16_t*>(Wuv), B,
                                                                         aa.n_split, out);
  return cudaGetLastError() == cudaSuccess ? SPC_OK : SPC_ERR_CUDA;
}

// ============================================================== latent gather
constexpr int kMgThreads = 512;
constexpr int kMgUnroll = 8;              // 16-byte pieces in flight per lane
constexpr int kMgSmsPerCta = 8;

// For host layers l in [layer_lo, layer_hi) of request b and load i:
//   slots[l - view.layer0, load_slot[b, i], :] = host[load_pos[b, i], l - view.store_layer0, :]
__global__ void __launch_bounds__(kMgThreads)
mla_gather_kernel(const spc_gather_view* __restrict__ views, int layer_lo, int layer_hi,
                  const int32_t* __restrict__ load_slot, const int32_t* __restrict__ load_pos,
                  const int32_t* __restrict__ n_load, int B, int K) {
  __shared__ int pre[SPC_MAX_BATCH + 1];
  __shared__ spc_gather_view sv[SPC_MAX_BATCH];
  const int tid = threadIdx.x;
  if (tid == 0) {
    int run = 0;
    for (int b = 0; b < B; ++b) { pre[b] = run; run += n_load[b]; }
    pre[B] = run;
  }
  for (int i = tid; i < B; i += kMgThreads) sv[i] = views[i];
  __syncthreads();
  const int R = pre[B];
  const int lane = tid & 31;
  const int w0 = (blockIdx.x * kMgThreads + tid) >> 5;
  const int nw = (gridDim.x * kMgThreads) >> 5;
  for (int j = w0; j < R; j += nw) {
    int b = 0;
    while (b + 1 < B && pre[b + 1] <= j) ++b;
    const int i = j - pre[b];
    const spc_gather_view vw = sv[b];
    const int l_begin = max(layer_lo, max(vw.layer0, vw.store_layer0));
    const int l_end = min(layer_hi, min(vw.layer0 + vw.n_layers, vw.store_layer0 + vw.store_layers));
    if (l_begin >= l_end) continue;
    const int pos = __ldg(load_pos + (size_t)b * K + i);
    const int slot = __ldg(load_slot + (size_t)b * K + i);
    // the run: every layer's latent row of this position, contiguous
    const uint16_t* run = static_cast<const uint16_t*>(vw.host) +
                          ((size_t)pos * vw.store_layers + (l_begin - vw.store_layer0)) * kLat;
    uint16_t* dst0 = static_cast<uint16_t*>(vw.slots) + ((size_t)(l_begin - vw.layer0) * K + slot) * kLat;
    const int n = (l_end - l_begin) * kLatPieces;
    for (int e0 = 0; e0 < n; e0 += 32 * kMgUnroll) {
      uint4 v[kMgUnroll];
#pragma unroll
      for (int u = 0; u < kMgUnroll; ++u) {
        const int e = e0 + lane + 32 * u;
        if (e < n) v[u] = ldg_stream(run + (size_t)e * 8);
      }
#pragma unroll
      for (int u = 0; u < kMgUnroll; ++u) {
        const int e = e0 + lane + 32 * u;
        if (e < n) {
          const int ly = e / kLatPieces, piece = e - ly * kLatPieces;
          stg_v4(dst0 + (size_t)ly * K * kLat + piece * 8, v[u]);
        }
      }
    }
  }
}

int mla_gather_launch(const spc_gather_view* views, int layer_lo, int layer_hi, const int32_t* load_slot,
                      const int32_t* load_pos, const int32_t* n_load, int B, int budget, void* stream) {
  if (layer_hi <= layer_lo) return SPC_OK;
  const long long per_block = kMgThreads / 32;
  long long grid = ((long long)B * budget + per_block - 1) / per_block;
  const long long cap_grid = std::max(4, device_sm_count() / kMgSmsPerCta);
  if (grid > cap_grid) grid = cap_grid;
  if (grid < 1) grid = 1;
  mla_gather_kernel<<<(int)grid, kMgThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      views, layer_lo, layer_hi, load_slot, load_pos, n_load, B, budget);
  return cudaGetLastError() == cudaSuccess ? SPC_OK : SPC_ERR_CUDA;
}

}  // namespace spc
