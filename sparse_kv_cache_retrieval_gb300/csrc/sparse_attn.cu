// Sparse GQA decode attention over the resident KV budget.
//
// Method: "ASPLOS'26 | SpeContext 让小模型先圈出重要 KV Cache" (marsggbo blog)
// §2 (softmax(QK^T/sqrt(d)) over the kept Top-K rows only) and §4 (the LLM
// forward runs on the sparse KV prepared in the previous iteration);
// "SpeContext: Enabling Efficient Long-context Reasoning with Speculative
// Context Sparsity in LLMs" (paperlayer.ai summary) §4.3 (for GQA the selected
// KV serves every query head of its group).
//
// GB300 design. Work item = a contiguous range of 64-row chunks of one
// (layer, request, KV head). Persistent CTAs of 4 consumer warps + 1 producer
// warp walk their items in a static round-robin:
//  * the producer streams each chunk's K and V rows into a 3-stage shared-
//    memory ring with cp.async.bulk (TMA engine, mbarrier byte counts): one
//    16 KiB copy per tensor in slot mode (slots are contiguous), one 256-byte
//    copy per kept row in position mode; it publishes a 64-bit mask of the
//    chunk's valid rows and runs ahead across item boundaries;
//  * consumers form the G heads' base-2 scores with a lane-rotated half-warp
//    reduce-scatter (each K row is read from shared memory once for the whole
//    group), update an online softmax per head (two named barriers per chunk),
//    and accumulate P.V in registers that persist across chunks, each thread
//    owning (heads, 8 columns) so a V row is read once per row group;
//  * an item's (max, sum, unnormalised output) is either the result or a
//    partial that the last CTA of its (layer, request, KV head) merges, in
//    split order (deterministic).
#include "spc_device.cuh"
#include "spc_internal.h"

namespace spc {

constexpr int kAttnRows = 64;                       // rows per chunk
constexpr int kAttnCWarps = 4;                      // consumer warps
constexpr int kAttnCThreads = kAttnCWarps * 32;     // 128
constexpr int kAttnThreads = kAttnCThreads + 32;    // + producer warp
constexpr int kAttnStages = 3;
constexpr uint32_t kAttnTileBytes = kAttnRows * kRowBytes;  // 16 KiB (K or V)
constexpr int kAttnItemsPerCta = 2;                 // split target: ~2 items per resident CTA
constexpr long long kAttnWait = 4000000000ll;
constexpr int kPartStride = kD + 4;                // (m, l, pad, pad, o[128])

template <int G>
struct AttnShape {
  static constexpr int HB = G < 8 ? G : 8;          // heads per register block
  static constexpr int NHB = G / HB;
  static constexpr int R = HB <= 4 ? 8 : 4;         // rows per half-warp QK batch
  static constexpr int NB = 8 / R;                  // batches (8 rows per half-warp per chunk)
  static constexpr int PAIRS = NHB * 16;            // (head block, 8-column chunk) pairs
  static constexpr int TPG = PAIRS < kAttnCThreads ? PAIRS : kAttnCThreads;
  static constexpr int RG = kAttnCThreads / TPG;    // row groups in P.V
  static constexpr int PPT = PAIRS / TPG;           // pairs per thread
  // row-group partial sums left after folding lanes l and l^16 (TPG <= 16)
  static constexpr int NRED = TPG <= 16 ? RG / 2 : RG;
  static constexpr int CTAS_PER_SM = G <= 8 ? 2 : 1;
};

struct AttnArgs {
  const uint16_t* q;
  const spc_kv_view* views;
  const int32_t* selected;
  const int32_t* slot_pos;
  float* out;
  float* part;
  uint32_t* counters;
  int* status;
  int B, n_q, n_kv, K, n_split, cps, n_chunks, n_items;
  float scale2;
};

template <int G>
struct AttnSmem {
  static constexpr size_t stages = (size_t)kAttnStages * 2 * kAttnTileBytes;
  static constexpr size_t q = sizeof(float) * G * kD;
  static constexpr size_t sc = sizeof(float) * G * kAttnRows;       // raw scores [G][64]
  static constexpr size_t pt = sizeof(float) * kAttnRows * G;       // weights [64][G]
  static constexpr size_t ored = sizeof(float) * AttnShape<G>::NRED * G * kD;
  static constexpr size_t small = sizeof(float) * 4 * 64 + sizeof(uint64_t) * (3 * kAttnStages);
  static constexpr size_t total = stages + q + sc + pt + ored + small;
};

__device__ __forceinline__ void cons_bar() { asm volatile("bar.sync 1, %0;" :: "n"(kAttnCThreads) : "memory"); }

template <int G>
__device__ __forceinline__ void item_coords(const AttnArgs& a, int item, int& lb, int& g, int& split) {
  split = item % a.n_split;
  const int rest = item / a.n_split;
  g = rest % a.n_kv;
  lb = rest / a.n_kv;
}

template <int G>
__global__ void __launch_bounds__(kAttnThreads) attn_kernel(AttnArgs a) {
  using S = AttnShape<G>;
  using M = AttnSmem<G>;
  extern __shared__ __align__(128) uint8_t asmem[];
  uint4* stage_kv = reinterpret_cast<uint4*>(asmem);                       // [stage][K|V][64][16]
  float* q_s = reinterpret_cast<float*>(asmem + M::stages);                // [G][128]
  float* sc = reinterpret_cast<float*>(asmem + M::stages + M::q);         // [G][64]
  float* pT = reinterpret_cast<float*>(asmem + M::stages + M::q + M::sc); // [64][G]
  float* ored = reinterpret_cast<float*>(asmem + M::stages + M::q + M::sc + M::pt);
  float* m_s = reinterpret_cast<float*>(asmem + M::stages + M::q + M::sc + M::pt + M::ored);
  float* l_s = m_s + 64;
  float* al_s = l_s + 64;
  uint64_t* okmask = reinterpret_cast<uint64_t*>(al_s + 128);
  uint64_t* full = okmask + kAttnStages;
  uint64_t* empty = full + kAttnStages;
  __shared__ int s_last;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kAttnStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kAttnCWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kAttnCWarps) {
    // ================= producer warp
    int it = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < a.n_items && ok; item += gridDim.x) {
      int lb, g, split;
      item_coords<G>(a, item, lb, g, split);
      const spc_kv_view vw = a.views[lb];
      const int b = lb % a.B;
      const int32_t* idx = (vw.use_slots ? a.slot_pos : a.selected) + ((size_t)b * a.n_kv + g) * a.K;
      const uint16_t* kb = static_cast<const uint16_t*>(vw.k) + (size_t)g * vw.rows * kD;
      const uint16_t* vb = static_cast<const uint16_t*>(vw.v) + (size_t)g * vw.rows * kD;
      const int c0 = split * a.cps, c1 = min(c0 + a.cps, a.n_chunks);
      for (int c = c0; c < c1; ++c, ++it) {
        const int s = it % kAttnStages;
        const uint32_t ph = (it / kAttnStages) & 1;
        if (!mbar_wait_bounded(&empty[s], ph ^ 1, kAttnWait)) {
          if (lane == 0) set_status(a.status, SPC_ERR_TIMEOUT);
          ok = false;
          break;
        }
        // row validity and source row for this lane's two rows
        int src[2];
        bool val[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int r = lane + 32 * h, i = c * kAttnRows + r;
          long long row = -1;
          if (i < a.K) {
            const int v = idx[i];
            if (v >= 0) row = vw.use_slots ? i : v;
            if (row >= vw.rows) row = -1;
          }
          val[h] = row >= 0;
          src[h] = (int)(row < 0 ? 0 : row);
        }
        const uint32_t lo = __ballot_sync(0xffffffffu, val[0]);
        const uint32_t hi = __ballot_sync(0xffffffffu, val[1]);
        uint4* kdst = stage_kv + (size_t)s * 2 * kAttnRows * 16;
        uint4* vdst = kdst + kAttnRows * 16;
        if (vw.use_slots) {
          // contiguous slots [c*64, min(K, c*64+64)): one copy per tensor
          const int n_in = min(kAttnRows, a.K - c * kAttnRows);
          if (lane == 0) {
            okmask[s] = ((uint64_t)hi << 32) | lo;
            mbar_arrive_expect_tx(&full[s], 2u * n_in * kRowBytes);
            bulk_g2s(kdst, kb + (size_t)c * kAttnRows * kD, n_in * kRowBytes, &full[s]);
            bulk_g2s(vdst, vb + (size_t)c * kAttnRows * kD, n_in * kRowBytes, &full[s]);
          }
        } else {
          const int nval = __popc(lo) + __popc(hi);
          if (lane == 0) {
            okmask[s] = ((uint64_t)hi << 32) | lo;
            mbar_arrive_expect_tx(&full[s], 2u * nval * kRowBytes);
          }
          __syncwarp();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (val[h]) {
              const int r = lane + 32 * h;
              bulk_g2s(kdst + r * 16, kb + (size_t)src[h] * kD, kRowBytes, &full[s]);
              bulk_g2s(vdst + r * 16, vb + (size_t)src[h] * kD, kRowBytes, &full[s]);
            }
          }
        }
        __syncwarp();
      }
    }
    // wait (bounded) for the copies still in flight before leaving
    if (lane == 0)
      for (int k = max(0, it - kAttnStages); k < it; ++k)
        mbar_wait_bounded(&full[k % kAttnStages], (k / kAttnStages) & 1, kAttnWait);
    return;
  }

  // ================= consumers (128 threads)
  const int ctid = tid;                        // 0..127
  const int hw = ctid >> 4, l16 = ctid & 15;   // half-warp 0..7 -> rows [hw*8, hw*8+8)
  const int rg = ctid / S::TPG, tp = ctid - rg * S::TPG;
  const int cc = tp & 15, hbp = tp >> 4;       // column chunk, first head block of this thread
  int it = 0;
  bool dead = false;  // a wait gave up: keep the barrier sequence, skip further waits
  for (int item = blockIdx.x; item < a.n_items; item += gridDim.x) {
    int lb, g, split;
    item_coords<G>(a, item, lb, g, split);
    const int c0 = split * a.cps, c1 = min(c0 + a.cps, a.n_chunks);

    // q of the group (base-2 scaled) and softmax state
    cons_bar();  // previous item's readers of q_s / m_s are done
    const uint16_t* qg = a.q + ((size_t)lb * a.n_q + (size_t)g * G) * kD;
    for (int i = ctid; i < G * kD; i += kAttnCThreads) q_s[i] = __uint_as_float(uint32_t(qg[i]) << 16) * a.scale2;
    for (int h = ctid; h < G; h += kAttnCThreads) { m_s[h] = -INFINITY; l_s[h] = 0.f; }
    cons_bar();
    float qr[S::HB][8];
    if (S::NHB == 1) {
#pragma unroll
      for (int h = 0; h < S::HB; ++h)
#pragma unroll
        for (int e = 0; e < 8; ++e) qr[h][e] = q_s[h * kD + l16 * 8 + e];
    }
    float acc[S::PPT][S::HB][8];
#pragma unroll
    for (int k = 0; k < S::PPT; ++k)
#pragma unroll
      for (int h = 0; h < S::HB; ++h)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[k][h][e] = 0.f;

    for (int c = c0; c < c1; ++c, ++it) {
      const int s = it % kAttnStages;
      const uint32_t ph = (it / kAttnStages) & 1;
      if (!dead && !mbar_wait_bounded(&full[s], ph, kAttnWait)) {
        if (lane == 0) set_status(a.status, SPC_ERR_TIMEOUT);
        dead = true;
      }
      const uint64_t okm = dead ? 0ull : okmask[s];
      const uint4* kt = stage_kv + (size_t)s * 2 * kAttnRows * 16;
      const uint4* vt = kt + kAttnRows * 16;

      // ---- scores, 8 rows per half-warp
#pragma unroll 1
      for (int hb = 0; hb < S::NHB; ++hb) {
        if (S::NHB > 1) {
#pragma unroll
          for (int h = 0; h < S::HB; ++h)
#pragma unroll
            for (int e = 0; e < 8; ++e) qr[h][e] = q_s[(hb * S::HB + h) * kD + l16 * 8 + e];
        }
#pragma unroll
        for (int bt = 0; bt < S::NB; ++bt) {
          const int rbase = hw * 8 + bt * S::R;
          float sacc[S::R][S::HB];
#pragma unroll
          for (int j = 0; j < S::R; ++j) {
            const uint4 w = kt[(rbase + (j ^ (l16 & (S::R - 1)))) * 16 + l16];
            float v[8];
            unpack8(w, v);
#pragma unroll
            for (int h = 0; h < S::HB; ++h) {
              float d0 = v[0] * qr[h][0];
#pragma unroll
              for (int e = 1; e < 8; ++e) d0 = fmaf(v[e], qr[h][e], d0);
              sacc[j][h] = d0;
            }
          }
#pragma unroll
          for (int m = S::R / 2; m >= 1; m >>= 1)
#pragma unroll
            for (int j = 0; j < m; ++j)
#pragma unroll
              for (int h = 0; h < S::HB; ++h) sacc[j][h] += __shfl_xor_sync(0xffffffffu, sacc[j + m][h], m);
#pragma unroll
          for (int m = S::R; m < 16; m <<= 1)
#pragma unroll
            for (int h = 0; h < S::HB; ++h) sacc[0][h] += __shfl_xor_sync(0xffffffffu, sacc[0][h], m);
          if (l16 < S::R) {
            const int r = rbase + l16;
            const bool ok = (okm >> r) & 1ull;
#pragma unroll
            for (int h = 0; h < S::HB; ++h) sc[(hb * S::HB + h) * kAttnRows + r] = ok ? sacc[0][h] : -INFINITY;
          }
        }
      }
      cons_bar();

      // ---- online softmax, heads spread over the 4 consumer warps
      for (int h = warp; h < G; h += kAttnCWarps) {
        const float x0 = sc[h * kAttnRows + lane], x1 = sc[h * kAttnRows + lane + 32];
        const float mo = m_s[h];
        const float mn = fmaxf(mo, warp_max(fmaxf(x0, x1)));
        const float p0 = mn == -INFINITY ? 0.f : exp2f(x0 - mn);
        const float p1 = mn == -INFINITY ? 0.f : exp2f(x1 - mn);
        pT[lane * G + h] = p0;
        pT[(lane + 32) * G + h] = p1;
        const float ps = warp_sum(p0 + p1);
        if (lane == 0) {
          const float alpha = (mn == -INFINITY) ? 1.f : exp2f(mo - mn);
          al_s[h] = alpha;
          l_s[h] = l_s[h] * alpha + ps;
          m_s[h] = mn;
        }
      }
      cons_bar();

      // ---- P.V over the valid rows of this thread's row group
#pragma unroll
      for (int k = 0; k < S::PPT; ++k) {
        const int h0 = (hbp + k * (S::TPG / 16)) * S::HB;
#pragma unroll
        for (int h = 0; h < S::HB; ++h) {
          const float al = al_s[h0 + h];
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[k][h][e] *= al;
        }
      }
      for (int r = rg; r < kAttnRows; r += S::RG) {
        if (!((okm >> r) & 1ull)) continue;
        const uint4 w = vt[r * 16 + cc];
        float v[8];
        unpack8(w, v);
#pragma unroll
        for (int k = 0; k < S::PPT; ++k) {
          const int h0 = (hbp + k * (S::TPG / 16)) * S::HB;
          float p[S::HB];
#pragma unroll
          for (int h = 0; h < S::HB; ++h) p[h] = pT[r * G + h0 + h];
#pragma unroll
          for (int h = 0; h < S::HB; ++h)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[k][h][e] = fmaf(p[h], v[e], acc[k][h][e]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }

    // ---- fold row groups (lanes l, l^16 in the warp, then the warps in a
    // fixed order); write the output or this split's partial
    if (S::TPG <= 16) {
#pragma unroll
      for (int k = 0; k < S::PPT; ++k)
#pragma unroll
        for (int h = 0; h < S::HB; ++h)
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[k][h][e] += __shfl_xor_sync(0xffffffffu, acc[k][h][e], 16);
    }
    if (S::TPG > 16 || lane < 16) {
      const int slot = S::TPG <= 16 ? warp : rg;
#pragma unroll
      for (int k = 0; k < S::PPT; ++k) {
        const int h0 = (hbp + k * (S::TPG / 16)) * S::HB;
#pragma unroll
        for (int h = 0; h < S::HB; ++h) {
          float* dst = ored + ((size_t)slot * G + h0 + h) * kD + cc * 8;
#pragma unroll
          for (int e = 0; e < 8; ++e) dst[e] = acc[k][h][e];
        }
      }
    }
    cons_bar();
    const size_t lbg = (size_t)lb * a.n_kv + g;
    float* outp = a.out + ((size_t)lb * a.n_q + (size_t)g * G) * kD;
    if (a.n_split == 1) {
      for (int i = ctid; i < G * kD; i += kAttnCThreads) {
        float o = 0.f;
#pragma unroll
        for (int r = 0; r < S::NRED; ++r) o += ored[(size_t)r * G * kD + i];
        const float l = l_s[i / kD];
        outp[i] = l > 0.f ? o / l : 0.f;
      }
      continue;
    }
    float* pp = a.part + (lbg * a.n_split + split) * (size_t)G * kPartStride;
    for (int i = ctid; i < G * kD; i += kAttnCThreads) {
      float o = 0.f;
#pragma unroll
      for (int r = 0; r < S::NRED; ++r) o += ored[(size_t)r * G * kD + i];
      pp[(i / kD) * kPartStride + 4 + (i % kD)] = o;
    }
    for (int h = ctid; h < G; h += kAttnCThreads) {
      pp[h * kPartStride] = m_s[h];
      pp[h * kPartStride + 1] = l_s[h];
    }
    __threadfence();
    cons_bar();
    if (ctid == 0) s_last = (atomicAdd(&a.counters[lbg], 1u) == (uint32_t)(a.n_split - 1));
    cons_bar();
    if (!s_last) continue;
    __threadfence();
    // merge the splits: stage every (max, sum) in shared memory (q_s is free
    // now), per head the global max and the weights, then float4 sums
    const float* pb = a.part + lbg * a.n_split * (size_t)G * kPartStride;
    float* wsp = q_s;                                   // [n_split][G] weights
    float* linv = q_s + a.n_split * G;                  // [G]
    for (int i = ctid; i < a.n_split * G; i += kAttnCThreads) wsp[i] = __ldcg(pb + (size_t)i * kPartStride);
    cons_bar();
    for (int h = ctid; h < G; h += kAttnCThreads) {
      float M = -INFINITY;
      for (int sp = 0; sp < a.n_split; ++sp) M = fmaxf(M, wsp[sp * G + h]);
      float Ls = 0.f;
      for (int sp = 0; sp < a.n_split; ++sp) {
        const float ms = wsp[sp * G + h];
        const float w = (M == -INFINITY || ms == -INFINITY) ? 0.f : exp2f(ms - M);
        Ls += __ldcg(pb + ((size_t)sp * G + h) * kPartStride + 1) * w;
        wsp[sp * G + h] = w;
      }
      linv[h] = Ls > 0.f ? 1.f / Ls : 0.f;
    }
    cons_bar();
    for (int i4 = ctid; i4 < G * (kD / 4); i4 += kAttnCThreads) {
      const int h = i4 / (kD / 4), c4 = i4 - h * (kD / 4);
      float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
      for (int sp = 0; sp < a.n_split; ++sp) {
        const float w = wsp[sp * G + h];
        const float4 v = __ldcg(reinterpret_cast<const float4*>(pb + ((size_t)sp * G + h) * kPartStride + 4) + c4);
        O.x = fmaf(w, v.x, O.x); O.y = fmaf(w, v.y, O.y); O.z = fmaf(w, v.z, O.z); O.w = fmaf(w, v.w, O.w);
      }
      const float li = linv[h];
      reinterpret_cast<float4*>(outp + (size_t)h * kD)[c4] = make_float4(O.x * li, O.y * li, O.z * li, O.w * li);
    }
    if (ctid == 0) a.counters[lbg] = 0u;
  }
}

static int attn_ctas_per_sm(int G) { return G <= 8 ? 2 : 1; }

static void attn_split(int n_layers, int B, int n_kv, int budget, int G, int* n_split, int* cps,
                       int* n_chunks) {
  const int nc = (budget + kAttnRows - 1) / kAttnRows;
  const long long base = (long long)n_layers * B * n_kv;
  // target items: ~2 per resident CTA on a 152-SM GB300 (a fixed count, so
  // the workspace size does not depend on the device)
  const long long target = (long long)kAttnItemsPerCta * attn_ctas_per_sm(G) * 152;
  long long want = (target + base - 1) / base;
  if (want < 1) want = 1;
  if (want > nc) want = nc;
  const int c = (int)((nc + want - 1) / want);
  *cps = c;
  *n_split = (nc + c - 1) / c;
  *n_chunks = nc;
}

size_t attn_workspace(int n_layers, int B, int n_q, int n_kv, int budget) {
  int ns, cps, nc;
  attn_split(n_layers, B, n_kv, budget, n_q / n_kv, &ns, &cps, &nc);
  const size_t nseg = (size_t)n_layers * B * n_kv;
  const size_t cnt = (nseg * sizeof(uint32_t) + 255) & ~size_t(255);
  const size_t part = ns > 1 ? nseg * ns * (size_t)(n_q / n_kv) * kPartStride * sizeof(float) : 0;
  return cnt + part;
}

template <int G>
static cudaError_t launch_attn(const AttnArgs& aa, cudaStream_t st) {
  const size_t smem = AttnSmem<G>::total;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(attn_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  int grid = AttnShape<G>::CTAS_PER_SM * device_sm_count();
  if (grid < 1) grid = 1;
  if (grid > aa.n_items) grid = aa.n_items;
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
  aa.status = nullptr;
  aa.B = B; aa.n_q = n_q; aa.n_kv = n_kv; aa.K = budget;
  attn_split(n_layers, B, n_kv, budget, n_q / n_kv, &aa.n_split, &aa.cps, &aa.n_chunks);
  aa.n_items = (int)(nseg * aa.n_split);
  aa.scale2 = scale * kLog2e;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  switch (n_q / n_kv) {
    case 1: e = launch_attn<1>(aa, st); break;
    case 2: e = launch_attn<2>(aa, st); break;
    case 4: e = launch_attn<4>(aa, st); break;
    case 8: e = launch_attn<8>(aa, st); break;
    case 16: e = launch_attn<16>(aa, st); break;
    case 32: e = launch_attn<32>(aa, st); break;
    default: e = launch_attn<64>(aa, st); break;
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
