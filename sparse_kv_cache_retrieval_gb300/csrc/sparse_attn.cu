// Sparse GQA decode attention over the resident KV budget.
//
// Method: "ASPLOS'26 | SpeContext 让小模型先圈出重要 KV Cache" (marsggbo blog)
// §2 (softmax(QK^T/sqrt(d)) over the kept Top-K rows only) and §4 (the LLM
// forward runs on the sparse KV prepared in the previous iteration);
// "SpeContext: Enabling Efficient Long-context Reasoning with Speculative
// Context Sparsity in LLMs" (paperlayer.ai summary) §4.3 (for GQA the selected
// KV serves every query head of its group).
//
// GB300 design. Per (layer, request, KV head) the kept rows form a small dense
// contraction: G query heads x 128 dims against up to `budget` rows. It is
// HBM-bound, but on CUDA cores its instruction stream (unpacking, shuffles,
// FMAs) held the SMs to ~1 instruction per cycle, well short of the memory
// rate. Here both products run on the tensor cores with mma.sync m16n8k16
// (bf16 in, fp32 accumulate; bf16 x bf16 products are exact in fp32):
//  * each (layer, request, KV head) is served by a thread-block cluster of up
//    to 8 CTAs (and, when a launch has too few of them to fill the GPU, by a
//    few such clusters); each CTA (4 consumer warps + 1 producer warp) streams
//    a contiguous range of 64-row chunks;
//  * the producer warp prefetches the CTA's row indices once, then copies each
//    chunk's K and V rows into a 3-stage shared-memory ring with 16-byte
//    cp.async (rows not kept are zero-filled), the 16-byte pieces of row r
//    placed at piece index ^ (r & 7) so that ldmatrix reads are free of bank
//    conflicts; cp.async completion arrives on the stage's mbarrier, and the
//    chunk's 64-bit valid-row mask is published with it;
//  * each consumer warp owns one 16-head tile of the group (zero-padded when
//    G < 16) and a slice of the chunk's rows: S = Q K^T from ldmatrix'ed K
//    fragments, masked online softmax in base 2 held per warp, then O += P V
//    with P reused from the S accumulators as an A fragment, split into bf16
//    high and low parts (two MMAs) so the weights keep ~16 bits, against
//    ldmatrix.trans'ed V fragments;
//  * warps sharing a head tile merge (max, sum, O) through shared memory; the
//    CTAs of a cluster merge through distributed shared memory (rank 0 reads
//    its peers); when several clusters share a (layer, request, KV head), each
//    writes a partial to the workspace and the last one merges them in split
//    order. Every merge is in a fixed order (deterministic).
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include <atomic>

#include "spc_device.cuh"
#include "spc_internal.h"

namespace spc {

constexpr int kAttnRows = 64;                       // rows per chunk
constexpr int kAttnPitch = 256;                     // smem bytes per row (16-byte chunks XOR-swizzled)
constexpr int kAttnCWarps = 4;
constexpr int kAttnCThreads = kAttnCWarps * 32;
constexpr int kAttnThreads = kAttnCThreads + 32;    // + producer warp
// ring depth: 2 stages for groups of up to 16 heads, so that two CTAs share
// an SM (their consumer warps hide each other's latency: at G = 8, 16 layers,
// 392 vs 605 us with 3 stages and one CTA per SM, the same with 4 or 6), 3
// for larger groups (whose merge buffers keep them at one CTA per SM)
template <int G>
constexpr int attn_stages() { return G <= 16 ? 2 : 3; }
constexpr int kAttnMaxCpc = 16;                     // chunks per CTA (row indices prefetched)
constexpr int kAttnTile = kAttnRows * kAttnPitch;   // 16 KiB (K or V)
constexpr int kAttnMaxCluster = 8;
constexpr int kAttnTargetCtas = 228;               // ~1.5 CTAs per SM of a 152-SM GB300
constexpr int kAttnWaveCtas = 304;                 // two CTAs per SM on 152 SMs
constexpr long long kAttnWait = 4000000000ll;
constexpr int kPartStride = kD + 4;                 // (m, l, pad, pad, o[128])

template <int G>
struct AttnShape {
  static constexpr int NMT = G <= 16 ? 1 : G / 16;  // 16-head tiles
  static constexpr int NRS = kAttnCWarps / NMT;     // warps sharing a tile (row split)
  static constexpr int RW = kAttnRows / NRS;        // rows per warp per chunk
  static constexpr int NT = RW / 8;                 // QK n-tiles (8 rows each)
  static constexpr int KS = RW / 16;                // PV k-steps (16 rows each)
  static constexpr int ST = attn_stages<G>();       // ring stages
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
  int B, n_q, n_kv, K, n_split, C, cpc, n_chunks;
  float scale2;
  long long wait_limit;   // clock cycles a bounded wait spends before it gives up
  int starve;             // test builds only: the producer issues no copies
};

// Workspace layout: a 256-byte status area (its first int32 is the status
// word), the per-(layer, request, KV head) merge counters, the split partials.
constexpr size_t kAttnStatusBytes = 256;

constexpr size_t round16(size_t x) { return (x + 15) & ~size_t(15); }

template <int G>
struct AttnSmem {
  using S = AttnShape<G>;
  static constexpr size_t stages = (size_t)S::ST * 2 * kAttnTile;
  static constexpr size_t mo = round16(sizeof(float) * S::NRS * G * kD);   // per row-split O
  static constexpr size_t ml = round16(sizeof(float) * 2 * S::NRS * G);    // per row-split (m, l)
  // row-split weights [NRS][G], later cluster weights [C][G] + sums [G]
  static constexpr size_t wsp = round16(sizeof(float) * ((S::NRS > kAttnMaxCluster ? S::NRS : kAttnMaxCluster) + 1) * G);
  static constexpr size_t cres = round16(sizeof(float) * G * kPartStride); // this CTA's (m, l, O)
  static constexpr size_t total = stages + mo + ml + wsp + cres + sizeof(uint64_t) * 3 * S::ST;
};

__device__ __forceinline__ void cons_bar() { asm volatile("bar.sync 1, %0;" :: "n"(kAttnCThreads) : "memory"); }

template <int G>
__global__ void __launch_bounds__(kAttnThreads) attn_kernel(AttnArgs a) {
  using S = AttnShape<G>;
  using M = AttnSmem<G>;
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ __align__(128) uint8_t asmem[];
  float* mo = reinterpret_cast<float*>(asmem + M::stages);                       // [NRS][G][128]
  float* ml = reinterpret_cast<float*>(asmem + M::stages + M::mo);               // [NRS][G][2]
  float* wsp = reinterpret_cast<float*>(asmem + M::stages + M::mo + M::ml);      // [NRS][G] + [G][2]
  float* cres = reinterpret_cast<float*>(asmem + M::stages + M::mo + M::ml + M::wsp);  // [G][132]
  uint64_t* okmask = reinterpret_cast<uint64_t*>(asmem + M::stages + M::mo + M::ml + M::wsp + M::cres);
  uint64_t* full = okmask + S::ST;
  uint64_t* empty = full + S::ST;
  __shared__ int s_last;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = (int)cluster.block_rank();
  const int cid = blockIdx.x / a.C;                 // cluster id
  const int split = cid % a.n_split, seg = cid / a.n_split;
  const int g = seg % a.n_kv, lb = seg / a.n_kv, b = lb % a.B;
  const int c0 = min(a.n_chunks, (split * a.C + rank) * a.cpc);
  const int c1 = min(a.n_chunks, c0 + a.cpc);

  if (tid == 0) {
    for (int s = 0; s < S::ST; ++s) {
      mbar_init(&full[s], 32 + 1);   // 32 cp.async arrivals + the mask publisher
      mbar_init(&empty[s], kAttnCWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kAttnCWarps) {
    // ================= producer warp: 16-byte cp.async into swizzled rows
    // row indices of every chunk of this CTA, two rows per lane per chunk,
    // fetched from both index arrays together with the view (one round trip)
    const spc_kv_view vw = a.views[lb];
    const size_t ioff = ((size_t)b * a.n_kv + g) * a.K;
    int srow[kAttnMaxCpc][2], ssel[kAttnMaxCpc][2];
#pragma unroll
    for (int k = 0; k < kAttnMaxCpc; ++k)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int i = (c0 + k) * kAttnRows + lane + 32 * h;
        const bool in = c0 + k < c1 && i < a.K;
        srow[k][h] = in ? a.slot_pos[ioff + i] : -1;
        ssel[k][h] = in ? a.selected[ioff + i] : -1;
      }
    if (!vw.use_slots) {
#pragma unroll
      for (int k = 0; k < kAttnMaxCpc; ++k) { srow[k][0] = ssel[k][0]; srow[k][1] = ssel[k][1]; }
    }
    const uint16_t* kb = static_cast<const uint16_t*>(vw.k) + (size_t)g * vw.rows * kD;
    const uint16_t* vb = static_cast<const uint16_t*>(vw.v) + (size_t)g * vw.rows * kD;
    int it = 0;
#ifdef SPC_TEST_HOOKS
    // a starved launch: no copy is issued and no stage is published, so every
    // consumer's first wait runs out (the path a lost copy would take)
    const int c_end = a.starve ? c0 : c1;
#else
    const int c_end = c1;
#endif
#pragma unroll 1
    for (int c = c0; c < c_end; ++c, ++it) {
      const int s = it % S::ST;
      const uint32_t ph = (it / S::ST) & 1;
      if (!mbar_wait_bounded(&empty[s], ph ^ 1, a.wait_limit)) {
        if (lane == 0) set_status(a.status, SPC_ERR_TIMEOUT);
        break;
      }
      bool val[2];
      int row[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        int v = -1;
#pragma unroll
        for (int k = 0; k < kAttnMaxCpc; ++k)
          if (k == it) v = srow[k][h];
        const int i = c * kAttnRows + lane + 32 * h;
        int r = -1;
        if (v >= 0) r = vw.use_slots ? i : v;
        if (r >= vw.rows) r = -1;
        val[h] = r >= 0;
        row[h] = r < 0 ? 0 : r;
      }
      const uint32_t lo = __ballot_sync(0xffffffffu, val[0]);
      const uint32_t hi = __ballot_sync(0xffffffffu, val[1]);
      uint8_t* kdst = asmem + (size_t)s * 2 * kAttnTile;
      uint8_t* vdst = kdst + kAttnTile;
      // one instruction copies two whole rows: lanes 0-15 row 2j, lanes 16-31
      // row 2j + 1, lane l its 16-byte piece l & 15 (coalesced 256-byte reads)
      const int piece = lane & 15, half = lane >> 4;
#pragma unroll 8
      for (int j = 0; j < kAttnRows / 2; ++j) {
        const int r = 2 * j + half;
        const int src_lane = r & 31;
        const int rr = __shfl_sync(0xffffffffu, j < 16 ? row[0] : row[1], src_lane);
        const uint32_t okw = j < 16 ? lo : hi;
        const int nb = ((okw >> src_lane) & 1u) ? 16 : 0;   // 0: zero-fill the row
        const int off = r * kAttnPitch + ((piece ^ (r & 7)) << 4);
        cp_async16(kdst + off, kb + (size_t)rr * kD + piece * 8, nb);
        cp_async16(vdst + off, vb + (size_t)rr * kD + piece * 8, nb);
      }
      if (lane == 0) {
        okmask[s] = ((uint64_t)hi << 32) | lo;
        mbar_arrive(&full[s]);
      }
      // arrives on full[s] once this lane's copies have landed
      asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" :: "r"(smem_u32(&full[s])) : "memory");
    }
    // wait (bounded) for the copies still in flight before leaving
    for (int k = max(0, it - S::ST); k < it; ++k)
      mbar_wait_bounded(&full[k % S::ST], (k / S::ST) & 1, a.wait_limit);
    __syncwarp();
  } else {
    // ================= consumers
    const int gid = lane >> 2, tig = lane & 3;
    const int mt = warp / S::NRS, rs = warp % S::NRS;
    const int row0 = rs * S::RW;                      // this warp's rows in a chunk
    const int h_lo = mt * 16 + gid, h_hi = h_lo + 8;  // heads of this thread's rows
    const uint32_t smem0 = smem_u32(asmem);
    const int lm = lane >> 3, lr = lane & 7;          // ldmatrix: matrix and row of this lane
    bool dead = false;

    // Q fragments of this warp's head tile (rows >= G are zero)
    const uint16_t* qg = a.q + ((size_t)lb * a.n_q + (size_t)g * G) * kD;
    uint32_t qf[8][4];
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int c = ks * 16 + tig * 2;
      qf[ks][0] = h_lo < G ? *reinterpret_cast<const uint32_t*>(qg + (size_t)h_lo * kD + c) : 0u;
      qf[ks][1] = h_hi < G ? *reinterpret_cast<const uint32_t*>(qg + (size_t)h_hi * kD + c) : 0u;
      qf[ks][2] = h_lo < G ? *reinterpret_cast<const uint32_t*>(qg + (size_t)h_lo * kD + c + 8) : 0u;
      qf[ks][3] = h_hi < G ? *reinterpret_cast<const uint32_t*>(qg + (size_t)h_hi * kD + c + 8) : 0u;
    }
    float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
    // P V layout. G <= 8 (kDM): O^T = V^T P^T with the 128 output dims on the
    // M side (8 m-tiles from ldmatrix.trans of the V rows) and P's bf16 high
    // and low parts packed on the N side (columns [0, HALF) high, [HALF,
    // 2 HALF) low, HALF = max(4, G)): 8 (G <= 4) or 16 (G = 8) MMAs per 16
    // keys. Larger groups keep heads on the M side (32 MMAs per 16 keys).
    constexpr bool kDM = G <= 8;
    constexpr int HALF = G < 4 ? 4 : G;
    constexpr int PNT = kDM ? (2 * HALF) / 8 : 1;
    float o[kDM ? 1 : 16][4];
    float oT[kDM ? 8 : 1][PNT][4];
#pragma unroll
    for (int n = 0; n < (kDM ? 1 : 16); ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
#pragma unroll
    for (int mt = 0; mt < (kDM ? 8 : 1); ++mt)
#pragma unroll
      for (int nt = 0; nt < PNT; ++nt) oT[mt][nt][0] = oT[mt][nt][1] = oT[mt][nt][2] = oT[mt][nt][3] = 0.f;

    int it = 0;
    for (int c = c0; c < c1; ++c, ++it) {
      const int s = it % S::ST;
      const uint32_t ph = (it / S::ST) & 1;
      if (!dead && !mbar_wait_bounded(&full[s], ph, a.wait_limit)) {
        if (lane == 0) set_status(a.status, SPC_ERR_TIMEOUT);
        dead = true;
      }
      const uint64_t okm = dead ? 0ull : okmask[s];
      const uint32_t kbase = smem0 + (uint32_t)(s * 2 * kAttnTile);
      const uint32_t vbase = kbase + kAttnTile;

      // ---- S = Q K^T over this warp's RW rows
      float sacc[S::NT][4];
#pragma unroll
      for (int n = 0; n < S::NT; ++n) sacc[n][0] = sacc[n][1] = sacc[n][2] = sacc[n][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
        for (int np = 0; np < S::NT / 2; ++np) {
          const int row = row0 + np * 16 + ((lm >> 1) << 3) + lr;
          const uint32_t addr = kbase + row * kAttnPitch + (((ks * 2 + (lm & 1)) ^ (row & 7)) << 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(addr, b0, b1, b2, b3);
          mma_bf16(sacc[2 * np], qf[ks], b0, b1);
          mma_bf16(sacc[2 * np + 1], qf[ks], b2, b3);
        }
      }
      // ---- masked online softmax (base 2), per head row of the tile
      float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
      for (int n = 0; n < S::NT; ++n) {
        const int r = row0 + n * 8 + tig * 2;
        const bool v0 = (okm >> r) & 1ull, v1 = (okm >> (r + 1)) & 1ull;
        sacc[n][0] = v0 ? sacc[n][0] * a.scale2 : -INFINITY;
        sacc[n][1] = v1 ? sacc[n][1] * a.scale2 : -INFINITY;
        sacc[n][2] = v0 ? sacc[n][2] * a.scale2 : -INFINITY;
        sacc[n][3] = v1 ? sacc[n][3] * a.scale2 : -INFINITY;
        mx_lo = fmaxf(mx_lo, fmaxf(sacc[n][0], sacc[n][1]));
        mx_hi = fmaxf(mx_hi, fmaxf(sacc[n][2], sacc[n][3]));
      }
#pragma unroll
      for (int off = 1; off <= 2; off <<= 1) {
        mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, off));
        mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, off));
      }
      const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
      const float al_lo = mn_lo == -INFINITY ? 1.f : exp2f(m_lo - mn_lo);
      const float al_hi = mn_hi == -INFINITY ? 1.f : exp2f(m_hi - mn_hi);
      float sum_lo = 0.f, sum_hi = 0.f;
#pragma unroll
      for (int n = 0; n < S::NT; ++n) {
        sacc[n][0] = mn_lo == -INFINITY ? 0.f : exp2f(sacc[n][0] - mn_lo);
        sacc[n][1] = mn_lo == -INFINITY ? 0.f : exp2f(sacc[n][1] - mn_lo);
        sacc[n][2] = mn_hi == -INFINITY ? 0.f : exp2f(sacc[n][2] - mn_hi);
        sacc[n][3] = mn_hi == -INFINITY ? 0.f : exp2f(sacc[n][3] - mn_hi);
        sum_lo += sacc[n][0] + sacc[n][1];
        sum_hi += sacc[n][2] + sacc[n][3];
      }
#pragma unroll
      for (int off = 1; off <= 2; off <<= 1) {
        sum_lo += __shfl_xor_sync(0xffffffffu, sum_lo, off);
        sum_hi += __shfl_xor_sync(0xffffffffu, sum_hi, off);
      }
      l_lo = l_lo * al_lo + sum_lo;
      l_hi = l_hi * al_hi + sum_hi;
      m_lo = mn_lo;
      m_hi = mn_hi;
      if (__any_sync(0xffffffffu, al_lo != 1.f || al_hi != 1.f)) {
        if constexpr (kDM) {
          // this lane's O^T columns 2tig, 2tig+1 belong to heads (2tig + e) mod HALF,
          // whose rescale factor sits in the lanes of row gid = head
          const float a0 = __shfl_sync(0xffffffffu, al_lo, ((2 * tig) & (HALF - 1)) * 4);
          const float a1 = __shfl_sync(0xffffffffu, al_lo, ((2 * tig + 1) & (HALF - 1)) * 4);
#pragma unroll
          for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int nt = 0; nt < PNT; ++nt) {
              oT[mt][nt][0] *= a0; oT[mt][nt][1] *= a1;
              oT[mt][nt][2] *= a0; oT[mt][nt][3] *= a1;
            }
        } else {
#pragma unroll
          for (int n = 0; n < 16; ++n) {
            o[n][0] *= al_lo; o[n][1] *= al_lo;
            o[n][2] *= al_hi; o[n][3] *= al_hi;
          }
        }
      }
      if constexpr (kDM) {
        // ---- O^T += V^T P^T. B fragment of column n = gid: keys (2tig, 2tig+1)
        // and (2tig+8, 2tig+9) of P's row for that column's head, which this
        // lane holds (row gid) for a high column; a low column of G <= 4 takes
        // the row of lane gid - 4 (lane ^ 16)
#pragma unroll
        for (int ks = 0; ks < S::KS; ++ks) {
          const float* p0 = sacc[2 * ks];
          const float* p1 = sacc[2 * ks + 1];
          uint32_t bh[2][PNT];
          if constexpr (PNT == 1) {
            const float y00 = __shfl_xor_sync(0xffffffffu, p0[0], 16), y01 = __shfl_xor_sync(0xffffffffu, p0[1], 16);
            const float y10 = __shfl_xor_sync(0xffffffffu, p1[0], 16), y11 = __shfl_xor_sync(0xffffffffu, p1[1], 16);
            if (gid < 4) {
              bh[0][0] = pack_bf16(bf16_round(p0[0]), bf16_round(p0[1]));
              bh[1][0] = pack_bf16(bf16_round(p1[0]), bf16_round(p1[1]));
            } else {
              bh[0][0] = pack_bf16(y00 - bf16_round(y00), y01 - bf16_round(y01));
              bh[1][0] = pack_bf16(y10 - bf16_round(y10), y11 - bf16_round(y11));
            }
          } else {
            const float h00 = bf16_round(p0[0]), h01 = bf16_round(p0[1]);
            const float h10 = bf16_round(p1[0]), h11 = bf16_round(p1[1]);
            bh[0][0] = pack_bf16(h00, h01);
            bh[1][0] = pack_bf16(h10, h11);
            bh[0][1] = pack_bf16(p0[0] - h00, p0[1] - h01);
            bh[1][1] = pack_bf16(p1[0] - h10, p1[1] - h11);
          }
          const int krow = row0 + ks * 16 + (lane & 7) + (((lane >> 4) & 1) << 3);
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            const int piece = mt * 2 + ((lane >> 3) & 1);
            uint32_t af[4];
            ldsm_x4_t(vbase + krow * kAttnPitch + ((piece ^ (krow & 7)) << 4), af[0], af[1], af[2], af[3]);
#pragma unroll
            for (int nt = 0; nt < PNT; ++nt) mma_bf16(oT[mt][nt], af, bh[0][nt], bh[1][nt]);
          }
        }
      } else {
      // ---- O += P V, P split into bf16 high + low parts
#pragma unroll
      for (int ks = 0; ks < S::KS; ++ks) {
        uint32_t ah[4], al[4];
        const float* p0 = sacc[2 * ks];
        const float* p1 = sacc[2 * ks + 1];
        const float h00 = bf16_round(p0[0]), h01 = bf16_round(p0[1]), h02 = bf16_round(p0[2]),
                    h03 = bf16_round(p0[3]);
        const float h10 = bf16_round(p1[0]), h11 = bf16_round(p1[1]), h12 = bf16_round(p1[2]),
                    h13 = bf16_round(p1[3]);
        ah[0] = pack_bf16(h00, h01); ah[1] = pack_bf16(h02, h03);
        ah[2] = pack_bf16(h10, h11); ah[3] = pack_bf16(h12, h13);
        al[0] = pack_bf16(p0[0] - h00, p0[1] - h01); al[1] = pack_bf16(p0[2] - h02, p0[3] - h03);
        al[2] = pack_bf16(p1[0] - h10, p1[1] - h11); al[3] = pack_bf16(p1[2] - h12, p1[3] - h13);
        const int vrow = row0 + ks * 16 + ((lm & 1) << 3) + lr;
#pragma unroll
        for (int dp = 0; dp < 8; ++dp) {
          const uint32_t addr = vbase + vrow * kAttnPitch + (((dp * 2 + (lm >> 1)) ^ (vrow & 7)) << 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(addr, b0, b1, b2, b3);
          mma_bf16(o[2 * dp], ah, b0, b1);
          mma_bf16(o[2 * dp], al, b0, b1);
          mma_bf16(o[2 * dp + 1], ah, b2, b3);
          mma_bf16(o[2 * dp + 1], al, b2, b3);
        }
      }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }

    // ---- merge the row-split warps of each head tile into this CTA's result
    if (tig == 0) {
      if (h_lo < G) { ml[(rs * G + h_lo) * 2] = m_lo; ml[(rs * G + h_lo) * 2 + 1] = l_lo; }
      if (h_hi < G) { ml[(rs * G + h_hi) * 2] = m_hi; ml[(rs * G + h_hi) * 2 + 1] = l_hi; }
    }
    if constexpr (kDM) {
      // O[h][dim] = O^T[dim][high column of h] + O^T[dim][low column of h]
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float v;
          if constexpr (PNT == 1) v = oT[mt][0][j] + __shfl_xor_sync(0xffffffffu, oT[mt][0][j], 2);
          else v = oT[mt][0][j] + oT[mt][1][j];
          const int head = 2 * tig + (j & 1);
          const int dim = mt * 16 + gid + ((j >> 1) << 3);
          if (head < G) mo[((size_t)rs * G + head) * kD + dim] = v;
        }
      }
    } else
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      const int d0 = n * 8 + tig * 2;
      if (h_lo < G) {
        mo[((size_t)rs * G + h_lo) * kD + d0] = o[n][0];
        mo[((size_t)rs * G + h_lo) * kD + d0 + 1] = o[n][1];
      }
      if (h_hi < G) {
        mo[((size_t)rs * G + h_hi) * kD + d0] = o[n][2];
        mo[((size_t)rs * G + h_hi) * kD + d0 + 1] = o[n][3];
      }
    }
    cons_bar();
    float* wr = wsp;                   // [NRS][G] row-split weights
    for (int h = tid; h < G; h += kAttnCThreads) {
      float Mx = -INFINITY;
#pragma unroll
      for (int r = 0; r < S::NRS; ++r) Mx = fmaxf(Mx, ml[(r * G + h) * 2]);
      float Ls = 0.f;
#pragma unroll
      for (int r = 0; r < S::NRS; ++r) {
        const float mr = ml[(r * G + h) * 2];
        const float w = (Mx == -INFINITY || mr == -INFINITY) ? 0.f : exp2f(mr - Mx);
        wr[r * G + h] = w;
        Ls += ml[(r * G + h) * 2 + 1] * w;
      }
      cres[h * kPartStride] = Mx;
      cres[h * kPartStride + 1] = Ls;
    }
    cons_bar();
    for (int i = tid; i < G * kD; i += kAttnCThreads) {
      const int h = i / kD;
      float v = 0.f;
#pragma unroll
      for (int r = 0; r < S::NRS; ++r) v += mo[(size_t)r * G * kD + i] * wr[r * G + h];
      cres[h * kPartStride + 4 + (i % kD)] = v;
    }
  }

  // ================= cluster merge (distributed shared memory), all threads
  cluster.sync();
  if (rank == 0 && warp < kAttnCWarps) {
    float* outp = a.out + ((size_t)lb * a.n_q + (size_t)g * G) * kD;
    const size_t lbg = (size_t)lb * a.n_kv + g;
    float* res = (a.n_split == 1) ? nullptr : a.part + (lbg * a.n_split + split) * (size_t)G * kPartStride;
    // per head: max and weights of the cluster's CTAs (wsp is free here)
    float* wc = wsp;  // [C][G] then [G] sums
    for (int h = tid; h < G; h += kAttnCThreads) {
      // every peer's (max, sum) in flight at once
      float2 ml_r[kAttnMaxCluster];
#pragma unroll
      for (int r = 0; r < kAttnMaxCluster; ++r)
        ml_r[r] = r < a.C ? *reinterpret_cast<const float2*>(cluster.map_shared_rank(cres + h * kPartStride, r))
                          : make_float2(-INFINITY, 0.f);
      float Mx = -INFINITY;
#pragma unroll
      for (int r = 0; r < kAttnMaxCluster; ++r) Mx = fmaxf(Mx, ml_r[r].x);
      float Ls = 0.f;
#pragma unroll
      for (int r = 0; r < kAttnMaxCluster; ++r) {
        const float w = (Mx == -INFINITY || ml_r[r].x == -INFINITY) ? 0.f : exp2f(ml_r[r].x - Mx);
        if (r < a.C) wc[r * G + h] = w;
        Ls += ml_r[r].y * w;
      }
      wc[a.C * G + h] = Ls;
      if (res) { res[h * kPartStride] = Mx; res[h * kPartStride + 1] = Ls; }
    }
    cons_bar();
    for (int i4 = tid; i4 < G * (kD / 4); i4 += kAttnCThreads) {
      const int h = i4 / (kD / 4), c4 = i4 - h * (kD / 4);
      float4 v[kAttnMaxCluster];
#pragma unroll
      for (int r = 0; r < kAttnMaxCluster; ++r)
        if (r < a.C)
          v[r] = *reinterpret_cast<const float4*>(cluster.map_shared_rank(cres + h * kPartStride + 4 + 4 * c4, r));
      float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int r = 0; r < kAttnMaxCluster; ++r) {
        if (r >= a.C) break;
        const float w = wc[r * G + h];
        O.x = fmaf(w, v[r].x, O.x); O.y = fmaf(w, v[r].y, O.y); O.z = fmaf(w, v[r].z, O.z); O.w = fmaf(w, v[r].w, O.w);
      }
      if (res) {
        reinterpret_cast<float4*>(res + h * kPartStride + 4)[c4] = O;
      } else {
        const float L = wc[a.C * G + h];
        const float li = L > 0.f ? 1.f / L : 0.f;
        reinterpret_cast<float4*>(outp + (size_t)h * kD)[c4] = make_float4(O.x * li, O.y * li, O.z * li, O.w * li);
      }
    }
    if (res) {
      // several clusters serve this (layer, request, KV head): the last merges
      __threadfence();
      cons_bar();
      if (tid == 0) s_last = (atomicAdd(&a.counters[lbg], 1u) == (uint32_t)(a.n_split - 1));
      cons_bar();
      if (s_last) {
        __threadfence();
        const float* pb = a.part + lbg * a.n_split * (size_t)G * kPartStride;
        float* wsplit = mo;                                 // [n_split][G]
        float* linv = mo + a.n_split * G;                   // [G]
        for (int i = tid; i < a.n_split * G; i += kAttnCThreads) wsplit[i] = __ldcg(pb + (size_t)i * kPartStride);
        cons_bar();
        for (int h = tid; h < G; h += kAttnCThreads) {
          float Mx = -INFINITY;
          for (int sp = 0; sp < a.n_split; ++sp) Mx = fmaxf(Mx, wsplit[sp * G + h]);
          float Ls = 0.f;
          for (int sp = 0; sp < a.n_split; ++sp) {
            const float ms = wsplit[sp * G + h];
            const float w = (Mx == -INFINITY || ms == -INFINITY) ? 0.f : exp2f(ms - Mx);
            Ls += __ldcg(pb + ((size_t)sp * G + h) * kPartStride + 1) * w;
            wsplit[sp * G + h] = w;
          }
          linv[h] = Ls > 0.f ? 1.f / Ls : 0.f;
        }
        cons_bar();
        for (int i4 = tid; i4 < G * (kD / 4); i4 += kAttnCThreads) {
          const int h = i4 / (kD / 4), c4 = i4 - h * (kD / 4);
          float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
          for (int sp = 0; sp < a.n_split; ++sp) {
            const float w = wsplit[sp * G + h];
            const float4 v = __ldcg(reinterpret_cast<const float4*>(pb + ((size_t)sp * G + h) * kPartStride + 4) + c4);
            O.x = fmaf(w, v.x, O.x); O.y = fmaf(w, v.y, O.y); O.z = fmaf(w, v.z, O.z); O.w = fmaf(w, v.w, O.w);
          }
          const float li = linv[h];
          reinterpret_cast<float4*>(outp + (size_t)h * kD)[c4] = make_float4(O.x * li, O.y * li, O.z * li, O.w * li);
        }
        if (tid == 0) a.counters[lbg] = 0u;
      }
    }
  }
  // keep this CTA's shared memory alive until rank 0 has read it
  cluster.sync();
}

static void attn_plan(int n_layers, int B, int n_kv, int budget, int* C, int* n_split, int* cpc,
                      int* n_chunks) {
  const int nc = (budget + kAttnRows - 1) / kAttnRows;
  const long long nseg = (long long)n_layers * B * n_kv;
  // cluster size: the largest power of two (up to 8) that keeps the launch
  // within one wave of two CTAs per SM, so each CTA streams many chunks and
  // pays its prologue and merge once; a fixed CTA target (not the device's SM
  // count) keeps the workspace size a function of the shapes alone
  int c = 1;
  while (c < kAttnMaxCluster && c < nc && nseg * c * 2 <= kAttnWaveCtas) c *= 2;
  long long s = (kAttnTargetCtas + nseg * c - 1) / (nseg * c);
  const int smax = (nc + c - 1) / c;
  if (s < 1) s = 1;
  if (s > smax) s = smax;
  // at most kAttnMaxCpc chunks per CTA (their row indices are prefetched)
  while ((nc + s * c - 1) / (s * c) > kAttnMaxCpc) ++s;
  *C = c;
  *n_split = (int)s;
  *cpc = (nc + (int)s * c - 1) / ((int)s * c);
  *n_chunks = nc;
}

size_t attn_workspace(int n_layers, int B, int n_q, int n_kv, int budget) {
  const size_t nseg = (size_t)n_layers * B * n_kv;
  const size_t cnt = (nseg * sizeof(uint32_t) + 255) & ~size_t(255);
  if (n_q / n_kv == attn_tc_group()) return kAttnStatusBytes + cnt + attn_tc_extra_bytes(n_layers, B, n_kv, budget);
  int C, ns, cpc, nc;
  attn_plan(n_layers, B, n_kv, budget, &C, &ns, &cpc, &nc);
  const size_t part = ns > 1 ? nseg * ns * (size_t)(n_q / n_kv) * kPartStride * sizeof(float) : 0;
  return kAttnStatusBytes + cnt + part;
}

#ifdef SPC_TEST_HOOKS
// Test builds only: the next `g_starve_calls` launches run starved, with a
// wait limit of `g_starve_wait` clock cycles.
static std::atomic<int> g_starve_calls{0};
static std::atomic<long long> g_starve_wait{0};
#endif

template <int G>
static cudaError_t launch_attn(const AttnArgs& aa, int nseg, cudaStream_t st) {
  const size_t smem = AttnSmem<G>::total;
  cudaError_t e = set_func_attr((const void*)attn_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(nseg * aa.n_split * aa.C));
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = aa.C;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_kernel<G>, aa);
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
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  aa.status = reinterpret_cast<int*>(ws);
  aa.counters = reinterpret_cast<uint32_t*>(ws + kAttnStatusBytes);
  aa.part = reinterpret_cast<float*>(ws + kAttnStatusBytes + ((nseg * sizeof(uint32_t) + 255) & ~size_t(255)));
  aa.wait_limit = kAttnWait;
  aa.starve = 0;
#ifdef SPC_TEST_HOOKS
  {
    int n = g_starve_calls.load();
    while (n > 0 && !g_starve_calls.compare_exchange_weak(n, n - 1)) {
    }
    if (n > 0) {
      aa.starve = 1;
      aa.wait_limit = g_starve_wait.load();
    }
  }
#endif
  aa.B = B; aa.n_q = n_q; aa.n_kv = n_kv; aa.K = budget;
  if (n_q / n_kv == attn_tc_group()) {
    // 64 heads per KV head: both products on tcgen05 (attn_tc.cu)
    AttnTcCall c{};
    c.q = aa.q; c.views = views; c.selected = selected; c.slot_pos = slot_pos; c.out = out;
    c.part = aa.part; c.counters = aa.counters; c.status = aa.status;
    c.B = B; c.n_q = n_q; c.n_kv = n_kv; c.K = budget;
    c.scale2 = scale * kLog2e;
    c.wait_limit = aa.wait_limit;
    c.starve = aa.starve;
    return attn_tc_launch(c, n_layers, stream);
  }
  attn_plan(n_layers, B, n_kv, budget, &aa.C, &aa.n_split, &aa.cpc, &aa.n_chunks);
  aa.scale2 = scale * kLog2e;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  switch (n_q / n_kv) {
    case 1: e = launch_attn<1>(aa, (int)nseg, st); break;
    case 2: e = launch_attn<2>(aa, (int)nseg, st); break;
    case 4: e = launch_attn<4>(aa, (int)nseg, st); break;
    case 8: e = launch_attn<8>(aa, (int)nseg, st); break;
    case 16: e = launch_attn<16>(aa, (int)nseg, st); break;
    default: e = launch_attn<32>(aa, (int)nseg, st); break;
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
  // the status word and the split-merge counters must start at zero; the
  // partials are always written before they are read
  const size_t nseg = (size_t)n_layers * B * n_kv;
  if (cudaMemsetAsync(scratch, 0, kAttnStatusBytes + nseg * sizeof(uint32_t), static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return SPC_ERR_CUDA;
  return attn_launch(q, views, selected, slot_pos, n_layers, B, n_q, n_kv, budget, scale, out,
                     scratch, stream);
}

}  // namespace spc

#ifdef SPC_TEST_HOOKS
// Test builds only (compiled with -DSPC_TEST_HOOKS into a separate library,
// never into libspc.so): the next `calls` launches of the GQA attention kernel
// run starved -- the producer issues no copies -- and their bounded waits give
// up after `wait_cycles` clock cycles, so a test can check that a wait that
// runs out records SPC_ERR_TIMEOUT in the status word and returns.
extern "C" int spc_test_starve_attention(int calls, long long wait_cycles) {
  if (calls < 0 || wait_cycles < 1) return SPC_ERR_INVALID_ARG;
  spc::g_starve_wait.store(wait_cycles);
  spc::g_starve_calls.store(calls);
  return SPC_OK;
}
#endif
