// Retrieval head on GB300: Q/K projection, key scan with per-head logsumexp
// partials, GQA group score and forced-set + Top-K selection.
//
// Method: "ASPLOS'26 | SpeContext 让小模型先圈出重要 KV Cache" (marsggbo blog)
// §5 (C1 lightweight retrieval head: keep the Q/K projections and the
// attention weights; head-level selection; GQA takes an element-wise max over
// a group's query heads, then Top-K per group; MQA is one group) and §2
// (softmax(QK^T/sqrt(d)), Top-K under the KV budget); "SpeContext: Enabling
// Efficient Long-context Reasoning with Speculative Context Sparsity in LLMs"
// (paperlayer.ai summary) §4.3. Forced sinks + recent window: SparseSpec-L news
// post and the same summary §2.2.
//
// GB300 design:
//  * proj_kernel: split-K GEMV over [W_q | W_k] (HBM-bound on the weights at
//    small batch), 16-byte loads, deterministic last-block reduction of the
//    split partials; the appended key row is rounded to bf16 and written in
//    place.
//  * scan_kernel: persistent CTAs; one producer warp streams 32 KiB tiles of
//    128 consecutive key rows into a 3-stage shared-memory ring with
//    cp.async.bulk (TMA engine, mbarrier completion); 4 consumer warps form
//    the dot products on CUDA cores (q in registers, fp32 accumulate) with a
//    lane-rotated row order so that a half-warp reduce-scatter needs no
//    selects; base-2 logits go to scratch and per-warp (max, sum 2^(l-max))
//    partials give the logsumexp.
//  * lse_kernel / score_kernel / topk_kernel: logsumexp per head, the group
//    score and its order key for every position on the whole GPU with a
//    per-(request, KV head) histogram of the key's bits 30..20, then one CTA
//    per (request, KV head) that finds the threshold key (histogram bin, then
//    two refinement passes over the bin's candidates) and writes the selection
//    with an ordered compaction (ascending, ties to the lower position).
#include <cuda_bf16.h>
#include <math.h>

#include "spc_device.cuh"
#include "spc_internal.h"

namespace spc {

__device__ __forceinline__ int effective_len(const int32_t* len, int b, int append, int cap) {
  int L = len[b];
  L = L < 0 ? 0 : (L > cap ? cap : L);
  return (append && L < cap) ? L + 1 : L;
}

// ============================================================== projection
struct ProjArgs {
  const uint16_t* x;
  const uint16_t* Wq;
  const uint16_t* Wk;
  uint16_t* K_dlm;
  const int32_t* len;
  float* q_ws;
  float* q_out;
  float* part;
  uint32_t* counters;
  int* status;
  int B, H, Nq, Nk, Ntot, n_kv, cap, S, Hc;
};

constexpr int kProjThreads = 256;
constexpr int kProjTile = 128;
constexpr int kProjBB = 16;  // batch rows per block (grid.z covers B)

template <int BB>
__device__ __forceinline__ void proj_fma(float (&acc)[BB][8], const uint4& w, const float* xr) {
  float v[8];
  unpack8(w, v);
#pragma unroll
  for (int bb = 0; bb < BB; ++bb) {
    const float xv = xr[bb];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[bb][e] = fmaf(v[e], xv, acc[bb][e]);
  }
}

template <int BB>
__global__ void __launch_bounds__(kProjThreads) proj_kernel(ProjArgs a) {
  extern __shared__ float psm[];
  __shared__ int s_last;
  const int tile = blockIdx.x, split = blockIdx.y, b0 = blockIdx.z * BB;
  const int col0 = tile * kProjTile;
  const bool is_k = col0 >= a.Nq;
  const uint16_t* W = is_k ? a.Wk : a.Wq;
  const int ld = is_k ? a.Nk : a.Nq;
  const int wcol0 = is_k ? col0 - a.Nq : col0;
  const int r_begin = split * a.Hc;
  const int nr = max(0, min(a.H, r_begin + a.Hc) - r_begin);

  float* xs = psm;                       // [Hc][BB]
  float* red = psm + a.Hc * BB;          // [8 warps][BB][128]
  for (int i = threadIdx.x; i < nr * BB; i += kProjThreads) {
    const int r = i / BB, bb = i - r * BB, b = b0 + bb;
    xs[i] = (b < a.B) ? __uint_as_float(uint32_t(a.x[(size_t)b * a.H + r_begin + r]) << 16) : 0.f;
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, l16 = lane & 15;
  float acc[BB][8];
#pragma unroll
  for (int bb = 0; bb < BB; ++bb)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[bb][e] = 0.f;

  const uint16_t* wp = W + (size_t)r_begin * ld + wcol0 + l16 * 8;
  int r = warp * 2 + (lane >> 4);
  for (; r + 112 < nr; r += 128) {
    uint4 w[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) w[u] = ldg_stream(wp + (size_t)(r + 16 * u) * ld);
#pragma unroll
    for (int u = 0; u < 8; ++u) proj_fma<BB>(acc, w[u], xs + (r + 16 * u) * BB);
  }
  for (; r < nr; r += 16) proj_fma<BB>(acc, ldg_stream(wp + (size_t)r * ld), xs + r * BB);

  // the two half-warps hold the same 128 columns: fold them, then across warps
#pragma unroll
  for (int bb = 0; bb < BB; ++bb)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[bb][e] += __shfl_xor_sync(0xffffffffu, acc[bb][e], 16);
  if (lane < 16) {
#pragma unroll
    for (int bb = 0; bb < BB; ++bb) {
      float4* dst = reinterpret_cast<float4*>(red + (warp * BB + bb) * kProjTile + l16 * 8);
      dst[0] = make_float4(acc[bb][0], acc[bb][1], acc[bb][2], acc[bb][3]);
      dst[1] = make_float4(acc[bb][4], acc[bb][5], acc[bb][6], acc[bb][7]);
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < BB * kProjTile; i += kProjThreads) {
    const int bb = i / kProjTile, c = i - bb * kProjTile;
    if (b0 + bb >= a.B) continue;
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kProjThreads / 32; ++w) s += red[(w * BB + bb) * kProjTile + c];
    a.part[((size_t)split * a.B + b0 + bb) * a.Ntot + col0 + c] = s;
  }

  // deterministic cross-block reduction: the last split block of this tile
  // sums the partials in split order and writes the result
  __threadfence();
  __syncthreads();
  const int ctr = tile * gridDim.z + blockIdx.z;
  if (threadIdx.x == 0) s_last = (atomicAdd(&a.counters[ctr], 1u) == (uint32_t)(a.S - 1));
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int i = threadIdx.x; i < BB * kProjTile; i += kProjThreads) {
    const int bb = i / kProjTile, c = i - bb * kProjTile, b = b0 + bb;
    if (b >= a.B) continue;
    float s4[4] = {0.f, 0.f, 0.f, 0.f};
    const float* pc = a.part + (size_t)b * a.Ntot + col0 + c;
    const size_t st = (size_t)a.B * a.Ntot;
    int sp = 0;
    for (; sp + 4 <= a.S; sp += 4) {
      s4[0] += __ldcg(pc + (sp + 0) * st);
      s4[1] += __ldcg(pc + (sp + 1) * st);
      s4[2] += __ldcg(pc + (sp + 2) * st);
      s4[3] += __ldcg(pc + (sp + 3) * st);
    }
    for (; sp < a.S; ++sp) s4[0] += __ldcg(pc + sp * st);
    const float s = (s4[0] + s4[1]) + (s4[2] + s4[3]);
    if (!is_k) {
      a.q_ws[(size_t)b * a.Nq + col0 + c] = s;
      if (a.q_out) a.q_out[(size_t)b * a.Nq + col0 + c] = s;
    } else {
      const int g = wcol0 / kD;
      const int L = a.len[b];
      if (L >= 0 && L < a.cap) {
        const __nv_bfloat16 h = __float2bfloat16_rn(s);
        a.K_dlm[(((size_t)b * a.n_kv + g) * a.cap + L) * kD + c] = __bfloat16_as_ushort(h);
      } else if (c == 0) {
        set_status(a.status, SPC_ERR_OVERFLOW);
      }
    }
  }
  if (threadIdx.x == 0) a.counters[ctr] = 0u;
}

// ============================================================== key scan
struct ScanArgs {
  const uint16_t* K;
  const float* q;
  const int32_t* len;
  float* logits;
  float2* part;
  int* status;
  int n_q, n_kv, cap, n_tiles, total_tiles, append, n_parts;
  float qscale;
};

constexpr int kScanRows = 128;
constexpr int kScanCWarps = 4;
constexpr int kScanThreads = (kScanCWarps + 1) * 32;
constexpr int kScanStages = 3;
constexpr uint32_t kScanTileBytes = kScanRows * kRowBytes;
constexpr long long kWaitLimit = 4000000000ll;  // clock cycles (~2 s)

template <int G>
struct ScanShape {
  static constexpr int HB = G < 8 ? G : 8;         // heads per register block
  static constexpr int R = HB <= 4 ? 16 : 8;       // rows per half-warp batch
  static constexpr int NB = 16 / R;                // batches per half-warp per tile
  static constexpr int NHB = G / HB;
  static constexpr int PPT = kScanCWarps * NB;     // lse partials per tile
};

template <int G>
__global__ void __launch_bounds__(kScanThreads) scan_kernel(ScanArgs a) {
  using S = ScanShape<G>;
  extern __shared__ __align__(128) uint8_t scan_smem[];
  uint4* tiles = reinterpret_cast<uint4*>(scan_smem);
  uint64_t* full = reinterpret_cast<uint64_t*>(scan_smem + kScanStages * kScanTileBytes);
  uint64_t* empty = full + kScanStages;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kScanStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kScanCWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kScanCWarps) {
    // ---------------- producer: one lane issues the bulk copies
    if (lane != 0) return;
    int it = 0;
    for (int t = blockIdx.x; t < a.total_tiles; t += gridDim.x) {
      const int seg = t / a.n_tiles, tile = t - seg * a.n_tiles;
      const int b = seg / a.n_kv;
      const int L = effective_len(a.len, b, a.append, a.cap);
      const int row0 = tile * kScanRows;
      if (row0 >= L) continue;
      const int nrows = min(kScanRows, L - row0);
      const int s = it % kScanStages;
      const uint32_t ph = (it / kScanStages) & 1;
      if (!mbar_wait_bounded(&empty[s], ph ^ 1, kWaitLimit)) {
        set_status(a.status, SPC_ERR_TIMEOUT);
        break;
      }
      mbar_arrive_expect_tx(&full[s], nrows * kRowBytes);
      bulk_g2s(tiles + (size_t)s * kScanRows * 16, a.K + ((size_t)seg * a.cap + row0) * kD,
               nrows * kRowBytes, &full[s]);
      ++it;
    }
    // wait (bounded) until every copy issued has landed before leaving
    for (int k = max(0, it - kScanStages); k < it; ++k)
      mbar_wait_bounded(&full[k % kScanStages], (k / kScanStages) & 1, kWaitLimit);
    return;
  }

  // ---------------- consumers
  const int hwi = warp * 2 + (lane >> 4);  // half-warp 0..7 -> rows [hwi*16, hwi*16+16)
  const int l16 = lane & 15;
  float qr[S::HB][8];
  int cur_seg = -1;
  int it = 0;
  for (int t = blockIdx.x; t < a.total_tiles; t += gridDim.x) {
    const int seg = t / a.n_tiles, tile = t - seg * a.n_tiles;
    const int b = seg / a.n_kv, g = seg - b * a.n_kv;
    const int L = effective_len(a.len, b, a.append, a.cap);
    const int row0 = tile * kScanRows;
    if (row0 >= L) continue;
    const int nrows = min(kScanRows, L - row0);
    const int s = it % kScanStages;
    const uint32_t ph = (it / kScanStages) & 1;
    if (!mbar_wait_bounded(&full[s], ph, kWaitLimit)) {
      set_status(a.status, SPC_ERR_TIMEOUT);
      break;
    }
    const uint4* tb = tiles + (size_t)s * kScanRows * 16;
    const float* qg = a.q + ((size_t)b * a.n_q + (size_t)g * G) * kD + l16 * 8;

    for (int bt = 0; bt < S::NB; ++bt) {
#pragma unroll 1
      for (int hb = 0; hb < S::NHB; ++hb) {
        if (S::NHB > 1 || seg != cur_seg) {
#pragma unroll
          for (int h = 0; h < S::HB; ++h) {
            const float4 q0 = __ldg(reinterpret_cast<const float4*>(qg + (size_t)(hb * S::HB + h) * kD));
            const float4 q1 = __ldg(reinterpret_cast<const float4*>(qg + (size_t)(hb * S::HB + h) * kD + 4));
            qr[h][0] = q0.x * a.qscale; qr[h][1] = q0.y * a.qscale;
            qr[h][2] = q0.z * a.qscale; qr[h][3] = q0.w * a.qscale;
            qr[h][4] = q1.x * a.qscale; qr[h][5] = q1.y * a.qscale;
            qr[h][6] = q1.z * a.qscale; qr[h][7] = q1.w * a.qscale;
          }
        }
        float acc[S::R][S::HB];
        const int rbase = hwi * 16 + bt * S::R;
#pragma unroll
        for (int j = 0; j < S::R; ++j) {
          // lane l16 reads chunk l16 of row (j ^ l16): conflict-free, and the
          // reduce-scatter below then needs compile-time indices only
          const uint4 w = tb[(rbase + (j ^ (l16 & (S::R - 1)))) * 16 + l16];
          float v[8];
          unpack8(w, v);
#pragma unroll
          for (int h = 0; h < S::HB; ++h) {
            float d0 = v[0] * qr[h][0];
#pragma unroll
            for (int e = 1; e < 8; ++e) d0 = fmaf(v[e], qr[h][e], d0);
            acc[j][h] = d0;
          }
        }
        // reduce-scatter over rows: lane keeps row (j ^ l16) for j < m
#pragma unroll
        for (int m = S::R / 2; m >= 1; m >>= 1) {
#pragma unroll
          for (int j = 0; j < m; ++j)
#pragma unroll
            for (int h = 0; h < S::HB; ++h)
              acc[j][h] += __shfl_xor_sync(0xffffffffu, acc[j + m][h], m);
        }
        // lanes l16 and l16 ^ R.. hold the same row: finish over the rest
#pragma unroll
        for (int m = S::R; m < 16; m <<= 1)
#pragma unroll
          for (int h = 0; h < S::HB; ++h) acc[0][h] += __shfl_xor_sync(0xffffffffu, acc[0][h], m);

        const int rloc = rbase + (l16 & (S::R - 1));
        const bool own = (l16 < S::R) && (rloc < nrows);
#pragma unroll
        for (int h = 0; h < S::HB; ++h) {
          const int hq = g * G + hb * S::HB + h;
          if (own) a.logits[((size_t)b * a.n_q + hq) * a.cap + row0 + rloc] = acc[0][h];
          const float mm = warp_max(own ? acc[0][h] : -INFINITY);
          const float ss = warp_sum(own ? exp2f(acc[0][h] - mm) : 0.f);
          if (lane == h)
            a.part[((size_t)b * a.n_q + hq) * a.n_parts + (size_t)tile * S::PPT + warp * S::NB + bt] =
                make_float2(mm, ss);
        }
      }
    }
    cur_seg = seg;
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    ++it;
  }
}

// ============================================================== group score + Top-K
// Three small kernels replace one long-latency one:
//  * lse_kernel: one CTA per query head folds the scan's (max, sum) partials
//    into log2-sum-exp;
//  * score_kernel: every position of every (request, KV head) in parallel:
//    s = max_h (l_h - lse_h), p = 2^s, the monotone uint32 order key of p, and
//    a 2048-bin histogram of the key's bits 30..20 (block histogram in shared
//    memory, flushed to a per-segment global histogram);
//  * topk_kernel: one CTA per (request, KV head) finds the bin holding the
//    (K-|F|)-th largest key, refines the remaining 21 bits over the bin's
//    candidates (gathered in shared memory; global fallback for huge ties),
//    then writes the selection with an ordered two-pass compaction (ties at
//    the threshold key to the lower positions). It leaves the global
//    histogram zeroed for the next call.
constexpr int kHistBins = 2048;
constexpr int kScoreThreads = 256;
constexpr int kScorePos = 2048;        // positions per score block
constexpr int kTopkThreads = 1024;
constexpr int kCandMax = 8192;

struct SelArgs {
  const float* logits;
  const float2* part;
  float* lse2;
  uint32_t* keys;
  uint32_t* ghist;
  int32_t* len;
  float* scores_out;
  int32_t* selected;
  uint32_t* done;
  int B, n_q, n_kv, G, cap, K, n_sink, n_recent, append, n_parts, ppt, kstride;
};

__device__ __forceinline__ bool is_forced(int p, int L, int n_sink, int n_recent) {
  return p < n_sink || p >= L - n_recent;
}

__global__ void __launch_bounds__(256) lse_kernel(SelArgs a) {
  const int bh = blockIdx.x, b = bh / a.n_q;
  const int L = effective_len(a.len, b, a.append, a.cap);
  const int nv = ((L + kScanRows - 1) / kScanRows) * a.ppt;
  const float2* ph = a.part + (size_t)bh * a.n_parts;
  float m = -INFINITY, s = 0.f;
  for (int i = threadIdx.x; i < nv; i += 256) {
    const float2 v = __ldcg(ph + i);
    lse2_combine(m, s, v.x, v.y);
  }
  warp_lse2(m, s);
  __shared__ float sm[8], ss[8];
  if ((threadIdx.x & 31) == 0) { sm[threadIdx.x >> 5] = m; ss[threadIdx.x >> 5] = s; }
  __syncthreads();
  if (threadIdx.x == 0) {
    float M = -INFINITY, Sx = 0.f;
    for (int w = 0; w < 8; ++w) lse2_combine(M, Sx, sm[w], ss[w]);
    a.lse2[bh] = Sx > 0.f ? M + log2f(Sx) : INFINITY;
  }
}

template <int G>
__global__ void __launch_bounds__(kScoreThreads) score_kernel(SelArgs a) {
  const int seg = blockIdx.y, b = seg / a.n_kv, g = seg - b * a.n_kv;
  const int L = effective_len(a.len, b, a.append, a.cap);
  const int p0 = blockIdx.x * kScorePos;
  if (p0 >= L) return;
  __shared__ uint32_t hist[kHistBins];
  __shared__ float lse[G];
  const int tid = threadIdx.x, lane = tid & 31;
  for (int i = tid; i < kHistBins; i += kScoreThreads) hist[i] = 0u;
  for (int h = tid; h < G; h += kScoreThreads) lse[h] = a.lse2[(size_t)b * a.n_q + (size_t)g * G + h];
  __syncthreads();
  const float* lg = a.logits + ((size_t)b * a.n_q + (size_t)g * G) * a.cap;
  constexpr int PER = kScorePos / kScoreThreads;  // 8 positions per thread
  constexpr int HC = G < 8 ? G : 8;               // heads per batch of loads in flight
  float sc[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) sc[k] = -INFINITY;
  for (int h0 = 0; h0 < G; h0 += HC) {
    float v[HC][PER];
#pragma unroll
    for (int h = 0; h < HC; ++h)
#pragma unroll
      for (int k = 0; k < PER; ++k) {
        const int p = p0 + k * kScoreThreads + tid;
        v[h][k] = p < L ? __ldcg(lg + (size_t)(h0 + h) * a.cap + p) : -INFINITY;
      }
#pragma unroll
    for (int h = 0; h < HC; ++h)
#pragma unroll
      for (int k = 0; k < PER; ++k) sc[k] = fmaxf(sc[k], v[h][k] - lse[h0 + h]);
  }
  // order key of the group score p = 2^s in [0, 1]: its float bits + 1 (0 is
  // reserved for forced / absent positions). Probabilities spread over many
  // exponents, so the key's bits 30..20 make a fine first histogram.
  uint32_t key[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int pos = p0 + k * kScoreThreads + tid;
    key[k] = 0u;
    if (pos < L) {
      const float pr = exp2f(sc[k]);
      if (a.scores_out) a.scores_out[(size_t)seg * a.cap + pos] = pr;
      if (!is_forced(pos, L, a.n_sink, a.n_recent)) key[k] = __float_as_uint(pr) + 1u;
      a.keys[(size_t)seg * a.kstride + pos] = key[k];
    }
  }
  if (L > a.K) {
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int bin = key[k] ? int(key[k] >> 20) : kHistBins;
      const unsigned peers = __match_any_sync(0xffffffffu, bin);
      if (bin < kHistBins && lane == __ffs(peers) - 1) atomicAdd(&hist[bin], (uint32_t)__popc(peers));
    }
    __syncthreads();
    uint32_t* gh = a.ghist + (size_t)seg * kHistBins;
    for (int i = tid; i < kHistBins; i += kScoreThreads)
      if (hist[i]) atomicAdd(&gh[i], hist[i]);
  }
}

// Bin (scanning from the top) where the running count reaches `rem`, over
// `nbins` counts held in shared memory; returns (bin, rem - count above it).
// Every thread of the block calls it. nbins <= 2 * blockDim.x.
__device__ __forceinline__ void find_bin(const uint32_t* cnt, int nbins, int rem, int* scratch,
                                         int* s_bin, int* s_rem) {
  const int t = threadIdx.x;
  const int bA = nbins - 1 - 2 * t, bB = nbins - 2 - 2 * t;  // descending pair
  const int cA = bA >= 0 ? (int)cnt[bA] : 0, cB = bB >= 0 ? (int)cnt[bB] : 0;
  int tot;
  const int before = block_excl_scan(cA + cB, scratch, &tot);
  if (bA >= 0 && before < rem && before + cA >= rem) { *s_bin = bA; *s_rem = rem - before; }
  if (bB >= 0 && before + cA < rem && before + cA + cB >= rem) { *s_bin = bB; *s_rem = rem - before - cA; }
  __syncthreads();
}

// Keys of positions [4*i4, 4*i4 + 4) with positions >= L zeroed.
__device__ __forceinline__ void keys4(const uint4* k4, int i4, int L, uint32_t k[4]) {
  const uint4 v = k4[i4];
  const int p = 4 * i4;
  k[0] = p + 0 < L ? v.x : 0u;
  k[1] = p + 1 < L ? v.y : 0u;
  k[2] = p + 2 < L ? v.z : 0u;
  k[3] = p + 3 < L ? v.w : 0u;
}

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(SelArgs a) {
  const int seg = blockIdx.x, b = seg / a.n_kv;
  const int L = effective_len(a.len, b, a.append, a.cap);
  const int tid = threadIdx.x, lane = tid & 31;
  int32_t* out = a.selected + (size_t)seg * a.K;
  const uint4* k4 = reinterpret_cast<const uint4*>(a.keys + (size_t)seg * a.kstride);
  uint32_t* gh = a.ghist + (size_t)seg * kHistBins;
  __shared__ uint32_t hist[kHistBins];
  __shared__ uint32_t cand[kCandMax];
  __shared__ int scratch[33];
  __shared__ int s_bin, s_rem, s_cnt, s_last;
  const int n4 = (L + 3) / 4;

  if (L <= a.K) {
    for (int p = tid; p < a.K; p += kTopkThreads) out[p] = p < L ? p : -1;
  } else {
    const int Kp = a.K - (a.n_sink + a.n_recent);
    uint32_t T = 0xffffffffu;
    int need = 0;
    // global histogram of the top 11 bits -> shared memory; leave it zeroed
    for (int i = tid; i < kHistBins; i += kTopkThreads) { hist[i] = gh[i]; gh[i] = 0u; }
    if (tid == 0) s_cnt = 0;
    __syncthreads();
    if (Kp > 0) {
      find_bin(hist, kHistBins, Kp, scratch, &s_bin, &s_rem);
      const uint32_t b1 = (uint32_t)s_bin;
      int rem = s_rem;
      const bool local = (int)hist[b1] <= kCandMax;
      if (local) {
        for (int i0 = tid; i0 < n4; i0 += 4 * kTopkThreads) {
          uint32_t kk[4][4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int i4 = i0 + u * kTopkThreads;
            if (i4 < n4) keys4(k4, i4, L, kk[u]);
            else kk[u][0] = kk[u][1] = kk[u][2] = kk[u][3] = 0u;
          }
#pragma unroll
          for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (kk[u][j] && (kk[u][j] >> 20) == b1) {
                const int c = atomicAdd(&s_cnt, 1);
                if (c < kCandMax) cand[c] = kk[u][j];
              }
        }
      }
      __syncthreads();
      // two refinement passes: bits 19..10, then 9..0
      uint32_t prefix = b1 << 20, mask = 0xfff00000u;
      for (int pass = 0; pass < 2; ++pass) {
        const int shift = pass == 0 ? 10 : 0;
        const int nb = 1024;
        const uint32_t dmask = (uint32_t)nb - 1u;
        for (int i = tid; i < kHistBins; i += kTopkThreads) hist[i] = 0u;
        __syncthreads();
        if (local) {
          const int n = min(s_cnt, kCandMax);
          for (int base = 0; base < n; base += kTopkThreads) {
            const int i = base + tid;
            const uint32_t k = i < n ? cand[i] : 0u;
            const int d = (k && (k & mask) == prefix) ? int((k >> shift) & dmask) : nb;
            const unsigned peers = __match_any_sync(0xffffffffu, d);
            if (d < nb && lane == __ffs(peers) - 1) atomicAdd(&hist[d], (uint32_t)__popc(peers));
          }
        } else {
          for (int base = 0; base < n4; base += kTopkThreads) {
            const int i4 = base + tid;
            uint32_t kk[4] = {0u, 0u, 0u, 0u};
            if (i4 < n4) keys4(k4, i4, L, kk);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t k = kk[j];
              const int d = (k && (k & mask) == prefix) ? int((k >> shift) & dmask) : nb;
              const unsigned peers = __match_any_sync(0xffffffffu, d);
              if (d < nb && lane == __ffs(peers) - 1) atomicAdd(&hist[d], (uint32_t)__popc(peers));
            }
          }
        }
        __syncthreads();
        find_bin(hist, nb, rem, scratch, &s_bin, &s_rem);
        prefix |= (uint32_t)s_bin << shift;
        mask |= dmask << shift;
        rem = s_rem;
        __syncthreads();
      }
      T = prefix;
      need = rem;
    }
    // ordered compaction: thread t owns the contiguous quads [q0, q1)
    const int qpt = (n4 + kTopkThreads - 1) / kTopkThreads;
    const int q0 = min(n4, tid * qpt), q1 = min(n4, q0 + qpt);
    int nb_ = 0, ne_ = 0;
    for (int qb = q0; qb < q1; qb += 8) {
      uint32_t kk[8][4];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (qb + u < q1) keys4(k4, qb + u, L, kk[u]);
        else kk[u][0] = kk[u][1] = kk[u][2] = kk[u][3] = 0u;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int p = 4 * (qb + u) + j;
          if (qb + u >= q1 || p >= L) continue;
          const uint32_t k = kk[u][j];
          if (is_forced(p, L, a.n_sink, a.n_recent) || (k && k > T)) ++nb_;
          else if (Kp > 0 && k && k == T) ++ne_;
        }
    }
    int tb, te;
    const int base_b = block_excl_scan(nb_, scratch, &tb);
    const int base_e = block_excl_scan(ne_, scratch, &te);
    int o = base_b + min(base_e, need);
    int eq_seen = base_e;
    for (int qb = q0; qb < q1; qb += 8) {
      uint32_t kk[8][4];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (qb + u < q1) keys4(k4, qb + u, L, kk[u]);
        else kk[u][0] = kk[u][1] = kk[u][2] = kk[u][3] = 0u;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int p = 4 * (qb + u) + j;
          if (qb + u >= q1 || p >= L) continue;
          const uint32_t k = kk[u][j];
          bool sel = is_forced(p, L, a.n_sink, a.n_recent) || (k && k > T);
          if (!sel && Kp > 0 && k && k == T) {
            sel = eq_seen < need;
            ++eq_seen;
          }
          if (sel) {
            if (o < a.K) out[o] = p;
            ++o;
          }
        }
    }
  }

  if (a.append) {
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      s_last = (atomicAdd(a.done, 1u) == gridDim.x - 1);
    }
    __syncthreads();
    if (s_last) {
      __threadfence();
      for (int bb = tid; bb < a.B; bb += kTopkThreads) {
        const int L0 = a.len[bb];
        if (L0 >= 0 && L0 < a.cap) a.len[bb] = L0 + 1;
      }
      if (tid == 0) *a.done = 0u;
    }
  }
}

// ============================================================== host side
struct ScoreLayout {
  size_t status, done, counters, q, part_proj, logits, part_scan, lse, keys, hist, total;
  int S, Hc, n_col_tiles, bz, n_tiles, ppt, n_parts;
};

static int proj_splits(int H) {
  int S = H / 256;
  return S < 1 ? 1 : (S > 32 ? 32 : S);
}

static int scan_ppt(int G) { return kScanCWarps * ((G < 8 ? G : 8) <= 4 ? 1 : 2); }

static ScoreLayout score_layout(int B, int H, int n_q, int n_kv, int cap) {
  ScoreLayout l{};
  const int Nq = n_q * kD, Nk = n_kv * kD, Ntot = Nq + Nk;
  l.S = proj_splits(H);
  l.Hc = (H + l.S - 1) / l.S;
  l.n_col_tiles = Ntot / kProjTile;
  l.bz = (B + kProjBB - 1) / kProjBB;
  l.n_tiles = (cap + kScanRows - 1) / kScanRows;
  l.ppt = scan_ppt(n_q / n_kv);
  l.n_parts = l.n_tiles * l.ppt;
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = (off + bytes + 255) & ~size_t(255); return o; };
  l.status = take(2 * sizeof(int));
  l.done = l.status + sizeof(int);
  l.counters = take(sizeof(uint32_t) * (size_t)l.n_col_tiles * 4 /* grid.z <= 4 */);
  l.q = take(sizeof(float) * (size_t)B * Nq);
  l.part_proj = take(sizeof(float) * (size_t)l.S * B * Ntot);
  l.logits = take(sizeof(float) * (size_t)B * n_q * cap);
  l.part_scan = take(sizeof(float2) * (size_t)B * n_q * l.n_parts);
  l.lse = take(sizeof(float) * (size_t)B * n_q);
  l.keys = take(sizeof(uint32_t) * (size_t)B * n_kv * ((cap + 3) & ~3));
  l.hist = take(sizeof(uint32_t) * (size_t)B * n_kv * kHistBins);
  l.total = off;
  return l;
}

size_t score_select_workspace(int B, int H, int n_q, int n_kv, int cap) {
  return score_layout(B, H, n_q, n_kv, cap).total;
}

template <int G>
static cudaError_t launch_scan(const ScanArgs& sa, int grid, cudaStream_t st) {
  const size_t smem = kScanStages * kScanTileBytes + 2 * kScanStages * sizeof(uint64_t);
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(scan_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  scan_kernel<G><<<grid, kScanThreads, smem, st>>>(sa);
  return cudaGetLastError();
}

template <int BB>
static cudaError_t launch_proj(const ProjArgs& pa, dim3 grid, size_t smem, cudaStream_t st) {
  static size_t attr = 0;
  if (smem > attr) {
    cudaError_t e = cudaFuncSetAttribute(proj_kernel<BB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr = smem;
  }
  proj_kernel<BB><<<grid, kProjThreads, smem, st>>>(pa);
  return cudaGetLastError();
}

int score_select_launch(const ScoreSelectCall& c) {
  const ScoreLayout l = score_layout(c.B, c.H, c.n_q, c.n_kv, c.cap);
  uint8_t* ws = static_cast<uint8_t*>(c.workspace);
  cudaStream_t st = static_cast<cudaStream_t>(c.stream);
  const int G = c.n_q / c.n_kv;
  const int Nq = c.n_q * kD, Nk = c.n_kv * kD;
  int* status = reinterpret_cast<int*>(ws + l.status);
  cudaError_t e;

  // ---- projection
  if (c.stages & SPC_STAGE_PROJECT) {
    ProjArgs pa{};
    pa.x = static_cast<const uint16_t*>(c.x);
    pa.Wq = static_cast<const uint16_t*>(c.Wq);
    pa.Wk = static_cast<const uint16_t*>(c.Wk);
    pa.K_dlm = static_cast<uint16_t*>(c.K_dlm);
    pa.len = c.len;
    pa.q_ws = reinterpret_cast<float*>(ws + l.q);
    pa.q_out = c.q_out;
    pa.part = reinterpret_cast<float*>(ws + l.part_proj);
    pa.counters = reinterpret_cast<uint32_t*>(ws + l.counters);
    pa.status = status;
    pa.B = c.B; pa.H = c.H; pa.Nq = Nq; pa.Nk = Nk; pa.Ntot = Nq + Nk; pa.n_kv = c.n_kv;
    pa.cap = c.cap; pa.S = l.S; pa.Hc = l.Hc;
    const int n_tiles = (Nq + (c.append ? Nk : 0)) / kProjTile;
    const int bb = c.B <= 1 ? 1 : c.B <= 2 ? 2 : c.B <= 4 ? 4 : c.B <= 8 ? 8 : 16;
    const dim3 grid(n_tiles, l.S, (c.B + bb - 1) / bb);
    const size_t smem = sizeof(float) * ((size_t)l.Hc * bb + (kProjThreads / 32) * bb * kProjTile);
    switch (bb) {
      case 1: e = launch_proj<1>(pa, grid, smem, st); break;
      case 2: e = launch_proj<2>(pa, grid, smem, st); break;
      case 4: e = launch_proj<4>(pa, grid, smem, st); break;
      case 8: e = launch_proj<8>(pa, grid, smem, st); break;
      default: e = launch_proj<16>(pa, grid, smem, st); break;
    }
    if (e != cudaSuccess) return SPC_ERR_CUDA;
  }

  // ---- key scan
  if (c.stages & SPC_STAGE_SCAN) {
    ScanArgs sa{};
    sa.K = static_cast<const uint16_t*>(c.K_dlm);
    sa.q = reinterpret_cast<const float*>(ws + l.q);
    sa.len = c.len;
    sa.logits = reinterpret_cast<float*>(ws + l.logits);
    sa.part = reinterpret_cast<float2*>(ws + l.part_scan);
    sa.status = status;
    sa.n_q = c.n_q; sa.n_kv = c.n_kv; sa.cap = c.cap; sa.n_tiles = l.n_tiles;
    sa.total_tiles = c.B * c.n_kv * l.n_tiles; sa.append = c.append; sa.n_parts = l.n_parts;
    sa.qscale = kLog2e / sqrtf((float)kD);
    int grid = 2 * device_sm_count();
    if (grid < 1) grid = 1;
    if (grid > sa.total_tiles) grid = sa.total_tiles;
    switch (G) {
      case 1: e = launch_scan<1>(sa, grid, st); break;
      case 2: e = launch_scan<2>(sa, grid, st); break;
      case 4: e = launch_scan<4>(sa, grid, st); break;
      case 8: e = launch_scan<8>(sa, grid, st); break;
      case 16: e = launch_scan<16>(sa, grid, st); break;
      case 32: e = launch_scan<32>(sa, grid, st); break;
      default: e = launch_scan<64>(sa, grid, st); break;
    }
    if (e != cudaSuccess) return SPC_ERR_CUDA;
  }

  // ---- logsumexp, group score + histogram, Top-K
  if (c.stages & SPC_STAGE_SELECT) {
    SelArgs sa{};
    sa.logits = reinterpret_cast<const float*>(ws + l.logits);
    sa.part = reinterpret_cast<const float2*>(ws + l.part_scan);
    sa.lse2 = reinterpret_cast<float*>(ws + l.lse);
    sa.keys = reinterpret_cast<uint32_t*>(ws + l.keys);
    sa.ghist = reinterpret_cast<uint32_t*>(ws + l.hist);
    sa.len = c.len;
    sa.scores_out = c.scores_out;
    sa.selected = c.selected;
    sa.done = reinterpret_cast<uint32_t*>(ws + l.done);
    sa.B = c.B; sa.n_q = c.n_q; sa.n_kv = c.n_kv; sa.G = G; sa.cap = c.cap; sa.K = c.budget;
    sa.n_sink = c.n_sink; sa.n_recent = c.n_recent; sa.append = c.append;
    sa.n_parts = l.n_parts; sa.ppt = l.ppt; sa.kstride = (c.cap + 3) & ~3;
    lse_kernel<<<c.B * c.n_q, 256, 0, st>>>(sa);
    if (cudaGetLastError() != cudaSuccess) return SPC_ERR_CUDA;
    const dim3 sg((c.cap + kScorePos - 1) / kScorePos, c.B * c.n_kv);
    switch (G) {
      case 1: score_kernel<1><<<sg, kScoreThreads, 0, st>>>(sa); break;
      case 2: score_kernel<2><<<sg, kScoreThreads, 0, st>>>(sa); break;
      case 4: score_kernel<4><<<sg, kScoreThreads, 0, st>>>(sa); break;
      case 8: score_kernel<8><<<sg, kScoreThreads, 0, st>>>(sa); break;
      case 16: score_kernel<16><<<sg, kScoreThreads, 0, st>>>(sa); break;
      case 32: score_kernel<32><<<sg, kScoreThreads, 0, st>>>(sa); break;
      default: score_kernel<64><<<sg, kScoreThreads, 0, st>>>(sa); break;
    }
    if (cudaGetLastError() != cudaSuccess) return SPC_ERR_CUDA;
    topk_kernel<<<c.B * c.n_kv, kTopkThreads, 0, st>>>(sa);
    if (cudaGetLastError() != cudaSuccess) return SPC_ERR_CUDA;
  }
  return SPC_OK;
}

}  // namespace spc
