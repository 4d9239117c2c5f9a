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
//    small batch), 16-byte loads, up to 16 in flight per thread; the splits
//    of a column tile form one thread-block cluster and meet in rank 0's
//    shared memory (fixed order, deterministic); the appended key row is
//    rounded to bf16 and written in place.
//  * scan_kernel: each CTA takes a few consecutive key tiles; one producer warp streams 32 KiB tiles of
//    128 consecutive key rows into a 3-stage shared-memory ring with coalesced
//    16-byte cp.async (XOR-swizzled rows, mbarrier completion); 4 consumer
//    warps form S = Q K^T on tensor cores (mma.sync m16n8k16 bf16, fp32
//    accumulate, q split into bf16 high + low parts) from ldmatrix fragments;
//    base-2 logits go to scratch and per-warp (max, sum 2^(l-max)) partials
//    give the logsumexp.
//  * select_kernel: one thread-block cluster per (request, KV head) folds the
//    logsumexp of each head, forms the group score and its order key for
//    every position, finds the threshold key with a radix select whose
//    histograms meet through distributed shared memory, and writes the
//    selection with an ordered compaction (ascending, ties to the lower
//    position).
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <math.h>

#include "spc_device.cuh"
#include "spc_internal.h"

#include <algorithm>

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
  int* status;
  int B, H, Nq, Nk, Ntot, n_kv, cap, S, Hc;
  int latent;   // 1: the appended row is one MLA latent row [B][cap][Nk] (Nk = 576)
};

#ifndef SPC_PROJ_TC_MIN_BATCH
#define SPC_PROJ_TC_MIN_BATCH 4   // batches of at least this many requests project on tensor cores
#endif
constexpr long long kWaitLimit = 4000000000ll;  // bounded mbarrier waits: clock cycles (~2 s)
constexpr int kProjThreads = 256;
constexpr int kProjTile = 128;
constexpr int kProjMaxSplit = 16;

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

// One cluster of S CTAs per 128-column tile: rank r forms the partial product
// over hidden rows [r*Hc, (r+1)*Hc); rank 0 sums the S partials through
// distributed shared memory in rank order (deterministic) and writes the
// result.
template <int BB>
__global__ void __launch_bounds__(kProjThreads) proj_kernel(ProjArgs a) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ float psm[];
  const int split = (int)cluster.block_rank();
  const int tile = blockIdx.x / a.S, b0 = blockIdx.z * BB;
  const int col0 = tile * kProjTile;
  const bool is_k = col0 >= a.Nq;
  const uint16_t* W = is_k ? a.Wk : a.Wq;
  const int ld = is_k ? a.Nk : a.Nq;
  const int wcol0 = is_k ? col0 - a.Nq : col0;
  // a tile may reach past the last weight column (the 576-column MLA latent
  // row: the fifth tile has 64 columns); lanes past it read the tile's first
  // columns, and their sums are not stored
  const int ncol = min(kProjTile, ld - wcol0);
  const int r_begin = split * a.Hc;
  const int nr = max(0, min(a.H, r_begin + a.Hc) - r_begin);

  float* xs = psm;                       // [Hc][BB]
  float* red = psm + a.Hc * BB;          // [8 warps][BB][128]; [BB][128] partial after the fold
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

  // half-warp hw takes rows hw, hw + 16, ...; LD weight loads in flight
  constexpr int LD = BB <= 2 ? 16 : 8;
  const uint16_t* wp = W + (size_t)r_begin * ld + wcol0 + (l16 * 8 < ncol ? l16 * 8 : 0);
  int r = warp * 2 + (lane >> 4);
  for (; r + 16 * (LD - 1) < nr; r += 16 * LD) {
    uint4 w[LD];
#pragma unroll
    for (int u = 0; u < LD; ++u) w[u] = ldg_stream(wp + (size_t)(r + 16 * u) * ld);
#pragma unroll
    for (int u = 0; u < LD; ++u) proj_fma<BB>(acc, w[u], xs + (r + 16 * u) * BB);
  }
  for (; r < nr; r += 16) proj_fma<BB>(acc, ldg_stream(wp + (size_t)r * ld), xs + r * BB);

  // the two half-warps hold the same 128 columns: fold them, then the warps
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
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < kProjThreads / 32; ++w) sum += red[w * BB * kProjTile + i];
    red[i] = sum;   // only this thread reads element i of warp 0's slice
  }
  cluster.sync();

  if (split == 0) {
    for (int i = threadIdx.x; i < BB * kProjTile; i += kProjThreads) {
      const int bb = i / kProjTile, c = i - bb * kProjTile, b = b0 + bb;
      if (b >= a.B || c >= ncol) continue;
      float v[kProjMaxSplit];
#pragma unroll
      for (int q = 0; q < kProjMaxSplit; ++q) v[q] = q < a.S ? *cluster.map_shared_rank(red + i, q) : 0.f;
      float sum = 0.f;
#pragma unroll
      for (int q = 0; q < kProjMaxSplit; ++q) sum += v[q];
      if (!is_k) {
        a.q_ws[(size_t)b * a.Nq + col0 + c] = sum;
        if (a.q_out) a.q_out[(size_t)b * a.Nq + col0 + c] = sum;
      } else {
        const int g = wcol0 / kD;
        const int L = a.len[b];
        if (L >= 0 && L < a.cap) {
          const __nv_bfloat16 h = __float2bfloat16_rn(sum);
          const size_t at = a.latent ? ((size_t)b * a.cap + L) * a.Nk + wcol0 + c
                                     : (((size_t)b * a.n_kv + g) * a.cap + L) * kD + c;
          a.K_dlm[at] = __bfloat16_as_ushort(h);
        } else if (c == 0) {
          set_status(a.status, SPC_ERR_OVERFLOW);
        }
      }
    }
  }
  // peers keep their shared memory until rank 0 has read it
  cluster.sync();
}

// Tensor-core projection for batched head inputs: [x_b; ...] (16 requests,
// zero-padded) times a 128-column tile of [W_q | W_k] on mma.sync m16n8k16
// (bf16 operands, exact products, fp32 accumulation). A producer warp streams
// 64-row slices of the weight tile (16 KiB) and the matching 64 columns of x
// (2 KiB) into a 4-stage ring with cp.async, both XOR-swizzled by 16-byte
// piece so ldmatrix reads are conflict-free; each of 4 consumer warps owns 32
// columns. The splits over H of one column tile form a thread-block cluster
// and meet in rank 0's shared memory in rank order, as in proj_kernel.
constexpr int kPtcRows = 64;                          // hidden rows per stage
constexpr int kPtcStages = 4;
constexpr int kPtcWarps = 4;
constexpr int kPtcThreads = (kPtcWarps + 1) * 32;
constexpr uint32_t kPtcWBytes = kPtcRows * kProjTile * 2;   // 16 KiB of weights
constexpr uint32_t kPtcXBytes = 16 * kPtcRows * 2;          // 2 KiB of x (16 rows x 128 B)
constexpr uint32_t kPtcStageBytes = kPtcWBytes + kPtcXBytes;
constexpr size_t kPtcSmem = (size_t)kPtcStages * kPtcStageBytes + sizeof(float) * 16 * kProjTile +
                            2 * kPtcStages * sizeof(uint64_t);

__global__ void __launch_bounds__(kPtcThreads) proj_tc_kernel(ProjArgs a) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ __align__(128) uint8_t ptc_smem[];
  const int split = (int)cluster.block_rank();
  const int tile = blockIdx.x / a.S, b0 = blockIdx.z * 16;
  const int col0 = tile * kProjTile;
  const bool is_k = col0 >= a.Nq;
  const uint16_t* W = is_k ? a.Wk : a.Wq;
  const int ld = is_k ? a.Nk : a.Nq;
  const int wcol0 = is_k ? col0 - a.Nq : col0;
  const int r_begin = split * a.Hc;                       // a multiple of 8
  const int nr = max(0, min(a.H, r_begin + a.Hc) - r_begin);   // a multiple of 8
  const int n_chunks = (nr + kPtcRows - 1) / kPtcRows;

  uint8_t* ring = ptc_smem;
  float* red = reinterpret_cast<float*>(ring + kPtcStages * kPtcStageBytes);   // [16][128] partial
  uint64_t* full = reinterpret_cast<uint64_t*>(red + 16 * kProjTile);
  uint64_t* empty = full + kPtcStages;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPtcStages; ++s) {
      mbar_init(&full[s], 32);
      mbar_init(&empty[s], kPtcWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kPtcWarps) {
    // ---------------- producer: per stage 64 weight rows of 256 bytes (two
    // rows per cp.async instruction, piece p of row r at p ^ (r & 7)) and 16 x
    // rows of 128 bytes (piece p of row r at p ^ (r & 7)); rows past the
    // slice or the batch are zero-filled
    const int piece = lane & 15, half = lane >> 4;
    const uint16_t* src0 = W + (size_t)r_begin * ld + wcol0 + piece * 8;
    for (int c = 0; c < n_chunks; ++c) {
      const int s = c % kPtcStages;
      const uint32_t ph = (c / kPtcStages) & 1;
      if (!mbar_wait_bounded(&empty[s], ph ^ 1, kWaitLimit)) {
        if (lane == 0) set_status(a.status, SPC_ERR_TIMEOUT);
        break;
      }
      uint8_t* dst = ring + (size_t)s * kPtcStageBytes;
#pragma unroll 8
      for (int j = 0; j < kPtcRows / 2; ++j) {
        const int r = 2 * j + half, rg = c * kPtcRows + r;
        const bool ok = rg < nr;
        cp_async16(dst + r * kRowBytes + ((piece ^ (r & 7)) << 4), src0 + (size_t)(ok ? rg : 0) * ld, ok ? 16 : 0);
      }
      uint8_t* xdst = dst + kPtcWBytes;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int idx = lane + 32 * i, xr = idx >> 3, xpc = idx & 7;
        const int k = c * kPtcRows + xpc * 8;
        const bool ok = b0 + xr < a.B && k < nr;
        const uint16_t* xs = ok ? a.x + (size_t)(b0 + xr) * a.H + r_begin + k : a.x;
        cp_async16(xdst + xr * (kPtcRows * 2) + ((xpc ^ (xr & 7)) << 4), xs, ok ? 16 : 0);
      }
      asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" :: "r"(smem_u32(&full[s])) : "memory");
    }
    for (int c = max(0, n_chunks - kPtcStages); c < n_chunks; ++c)
      mbar_wait_bounded(&full[c % kPtcStages], (c / kPtcStages) & 1, kWaitLimit);
  } else {
    // ---------------- consumers: warp w owns columns [32w, 32w + 32)
    float acc[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    const int xr = lane & 15, xhi = lane >> 4;                 // A: x row and k-half this lane addresses
    const int krow = (lane & 7) + (((lane >> 3) & 1) << 3);    // B: weight row within a 16-row k-step
    const int npc = warp * 4 + (lane >> 4);                    // B: first 16-byte column piece
    for (int c = 0; c < n_chunks; ++c) {
      const int s = c % kPtcStages;
      const uint32_t ph = (c / kPtcStages) & 1;
      if (!mbar_wait_bounded(&full[s], ph, kWaitLimit)) {
        if (lane == 0) set_status(a.status, SPC_ERR_TIMEOUT);
        break;
      }
      const uint32_t wbase = smem_u32(ring + (size_t)s * kPtcStageBytes);
      const uint32_t xbase = wbase + kPtcWBytes + xr * (kPtcRows * 2);
#pragma unroll
      for (int ks = 0; ks < kPtcRows / 16; ++ks) {
        uint32_t af[4];
        ldsm_x4(xbase + (((ks * 2 + xhi) ^ (xr & 7)) << 4), af[0], af[1], af[2], af[3]);
        const int r = ks * 16 + krow;
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {
          const int pc = npc + pr * 2;
          uint32_t b00, b01, b10, b11;
          ldsm_x4_t(wbase + r * kRowBytes + ((pc ^ (r & 7)) << 4), b00, b01, b10, b11);
          mma_bf16(acc[2 * pr], af, b00, b01);
          mma_bf16(acc[2 * pr + 1], af, b10, b11);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    // this split's partial: rows gid / gid + 8, columns 32w + 8nt + 2tig (+1)
    const int gid = lane >> 2, tig = lane & 3;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int cc = warp * 32 + nt * 8 + tig * 2;
      *reinterpret_cast<float2*>(red + gid * kProjTile + cc) = make_float2(acc[nt][0], acc[nt][1]);
      *reinterpret_cast<float2*>(red + (gid + 8) * kProjTile + cc) = make_float2(acc[nt][2], acc[nt][3]);
    }
  }
  cluster.sync();

  if (split == 0) {
    for (int i = threadIdx.x; i < 16 * kProjTile; i += kPtcThreads) {
      const int bb = i / kProjTile, c = i - bb * kProjTile, b = b0 + bb;
      if (b >= a.B) continue;
      float v[kProjMaxSplit];
#pragma unroll
      for (int q = 0; q < kProjMaxSplit; ++q) v[q] = q < a.S ? *cluster.map_shared_rank(red + i, q) : 0.f;
      float sum = 0.f;
#pragma unroll
      for (int q = 0; q < kProjMaxSplit; ++q) sum += v[q];
      if (!is_k) {
        a.q_ws[(size_t)b * a.Nq + col0 + c] = sum;
        if (a.q_out) a.q_out[(size_t)b * a.Nq + col0 + c] = sum;
      } else {
        const int g = wcol0 / kD;
        const int L = a.len[b];
        if (L >= 0 && L < a.cap) {
          const __nv_bfloat16 h = __float2bfloat16_rn(sum);
          a.K_dlm[(((size_t)b * a.n_kv + g) * a.cap + L) * kD + c] = __bfloat16_as_ushort(h);
        } else if (c == 0) {
          set_status(a.status, SPC_ERR_OVERFLOW);
        }
      }
    }
  }
  cluster.sync();
}

// ============================================================== key scan
struct ScanArgs {
  const uint16_t* K;
  const float* q;
  const int32_t* len;
  float* logits;
  float2* part;
  int* status;
  int n_q, n_kv, cap, lstride, n_tiles, total_tiles, append, n_parts, tpc;
  float qscale;
};

constexpr int kScanRows = 128;
constexpr int kScanStages = 3;
// Tiles per CTA: 0 sizes the grid to one wave of kScanCtasPerSm CTAs per SM
// (each CTA streams a run of consecutive tiles, so the kernel lasts as long
// as its longest run); a positive value fixes the run length.
#ifndef SPC_SCAN_TILES_PER_CTA
#define SPC_SCAN_TILES_PER_CTA 0
#endif
constexpr int kScanTilesPerCta = SPC_SCAN_TILES_PER_CTA;
constexpr int kScanCtasPerSm = 2;   // the 3-stage ring with its query copies (108 KB) allows two per SM
constexpr uint32_t kScanTileBytes = kScanRows * kRowBytes;
// fp32 queries of a group of up to 8 heads, copied by the producer with the
// first tile of each segment a CTA meets, into that tile's stage
constexpr uint32_t kScanQBytes = 8 * kD * 4;
constexpr size_t kScanSmem = (size_t)kScanStages * (kScanTileBytes + kScanQBytes) + 2 * kScanStages * sizeof(uint64_t);

// Key-major tensor-core scan for groups of up to 8 query heads. The key rows
// are the M side of m16n8k16 (16 keys x 16 dims per ldmatrix.x4 from the
// swizzled tile); the N side holds the group's queries twice, the bf16 high
// parts in columns [0, HALF) and the low parts in [HALF, 2*HALF), HALF =
// max(4, G), so one product yields both halves and their sum is q.K with
// about 16 significant bits in q. Per 128-key tile each of 8 consumer warps
// takes 16 keys: 8 (G <= 4) or 16 (G = 8) MMAs, two accumulator chains over
// the halves of the head dimension. The tile's stage is released as soon as
// its last fragment is in registers.
constexpr int kScanKmWarps = 8;
constexpr int kScanKmThreads = (kScanKmWarps + 1) * 32;

template <int G>
struct ScanKmShape {
  static constexpr int HALF = G < 4 ? 4 : G;   // columns per half (high / low)
  static constexpr int NT = 2 * HALF / 8;      // n-tiles of 8 columns
  static constexpr int PPT = kScanKmWarps;     // logsumexp partials per tile per head
};

template <int G>
__global__ void __launch_bounds__(kScanKmThreads) scan_kernel_km(ScanArgs a) {
  static_assert(G <= 8, "key-major scan serves groups of at most 8 heads");
  using S = ScanKmShape<G>;
  extern __shared__ __align__(128) uint8_t scan_smem[];
  uint8_t* qarea = scan_smem + kScanStages * kScanTileBytes;          // [kScanStages][kScanQBytes]
  uint64_t* full = reinterpret_cast<uint64_t*>(qarea + kScanStages * kScanQBytes);
  uint64_t* empty = full + kScanStages;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kScanStages; ++s) {
      mbar_init(&full[s], 32);       // one cp.async arrival per producer lane
      mbar_init(&empty[s], kScanKmWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  const int t_end = min(a.total_tiles, (blockIdx.x + 1) * a.tpc);

  if (warp == kScanKmWarps) {
    // ---------------- producer: as in scan_kernel (two rows per cp.async
    // instruction, piece p of row r stored at p ^ (r & 7), tail zero-filled)
    const int piece = lane & 15, half = lane >> 4;
    int it = 0, q_seg = -1;
    for (int t = blockIdx.x * a.tpc; t < t_end; ++t) {
      const int seg = t / a.n_tiles, tile = t - seg * a.n_tiles;
      const int b = seg / a.n_kv;
      const int L = effective_len(a.len, b, a.append, a.cap);
      const int row0 = tile * kScanRows;
      if (row0 >= L) continue;
      const int nrows = min(kScanRows, L - row0);
      const int s = it % kScanStages;
      const uint32_t ph = (it / kScanStages) & 1;
      if (!mbar_wait_bounded(&empty[s], ph ^ 1, kWaitLimit)) {
        if (lane == 0) set_status(a.status, SPC_ERR_TIMEOUT);
        break;
      }
      uint8_t* dst = scan_smem + (size_t)s * kScanTileBytes;
      if (seg != q_seg) {
        // the segment's queries ride with its first tile (loaded by the
        // consumers they would queue behind the ring's copies)
        const int g = seg - b * a.n_kv;
        const float* qg = a.q + ((size_t)b * a.n_q + (size_t)g * G) * kD;
        uint8_t* qd = qarea + (size_t)s * kScanQBytes;
#pragma unroll
        for (int j = 0; j < G; ++j) cp_async16(qd + (size_t)(lane + 32 * j) * 16, qg + (lane + 32 * j) * 4, 16);
        q_seg = seg;
      }
      const uint16_t* src = a.K + ((size_t)seg * a.cap + row0) * kD + piece * 8;
#pragma unroll 8
      for (int j = 0; j < kScanRows / 2; ++j) {
        const int r = 2 * j + half;
        const bool ok = r < nrows;
        cp_async16(dst + r * kRowBytes + ((piece ^ (r & 7)) << 4), src + (size_t)(ok ? r : 0) * kD, ok ? 16 : 0);
      }
      asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" :: "r"(smem_u32(&full[s])) : "memory");
      ++it;
    }
    for (int k = max(0, it - kScanStages); k < it; ++k)
      mbar_wait_bounded(&full[k % kScanStages], (k / kScanStages) & 1, kWaitLimit);
    return;
  }

  // ---------------- consumers
  const int gid = lane >> 2, tig = lane & 3, mi = lane >> 3, ri = lane & 7;
  const int r0 = warp * 16;                       // this warp's 16 keys of a tile
  const int hA = 2 * tig, hB = hA + 1;            // heads of this lane's C columns
  uint32_t qb[8][S::NT][2];                       // B fragments: q high / low, per k-step
  int cur_seg = -1;
  int it = 0;
  for (int t = blockIdx.x * a.tpc; t < t_end; ++t) {
    const int seg = t / a.n_tiles, tile = t - seg * a.n_tiles;
    const int b = seg / a.n_kv, g = seg - b * a.n_kv;
    const int L = effective_len(a.len, b, a.append, a.cap);
    const int row0 = tile * kScanRows;
    if (row0 >= L) continue;
    const int nrows = min(kScanRows, L - row0);
    const int s = it % kScanStages;
    const uint32_t ph = (it / kScanStages) & 1;
    if (!mbar_wait_bounded(&full[s], ph, kWaitLimit)) {
      if (lane == 0) set_status(a.status, SPC_ERR_TIMEOUT);
      break;
    }
    if (seg != cur_seg) {
      // this tile's stage holds the segment's queries (fp32 [G][128])
      const float* qg = reinterpret_cast<const float*>(qarea + (size_t)s * kScanQBytes);
      (void)g;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
        for (int nt = 0; nt < S::NT; ++nt) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int col = nt * 8 + gid;
            const bool low = col >= S::HALF;
            const int h = low ? col - S::HALF : col;
            const int k = ks * 16 + tig * 2 + e * 8;
            float2 v = make_float2(0.f, 0.f);
            if (h < G) v = *reinterpret_cast<const float2*>(qg + (size_t)h * kD + k);
            const float x = v.x * a.qscale, y = v.y * a.qscale;
            const float xh = bf16_round(x), yh = bf16_round(y);
            qb[ks][nt][e] = low ? pack_bf16(x - xh, y - yh) : pack_bf16(xh, yh);
          }
        }
      }
      cur_seg = seg;
    }
    const uint32_t base = smem_u32(scan_smem + (size_t)s * kScanTileBytes);
    float acc[2][S::NT][4];
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
      for (int nt = 0; nt < S::NT; ++nt) acc[c][nt][0] = acc[c][nt][1] = acc[c][nt][2] = acc[c][nt][3] = 0.f;
    const int row = r0 + ri + ((mi & 1) << 3);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int piece = ks * 2 + (mi >> 1);
      uint32_t af[4];
      ldsm_x4(base + row * kRowBytes + ((piece ^ (row & 7)) << 4), af[0], af[1], af[2], af[3]);
#pragma unroll
      for (int nt = 0; nt < S::NT; ++nt) mma_bf16(acc[ks & 1][nt], af, qb[ks][nt][0], qb[ks][nt][1]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);

    // high + low halves: l[0], l[1] = key r0+gid, heads hA, hB; l[2], l[3] = key r0+gid+8
    float l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float v[S::NT];
#pragma unroll
      for (int nt = 0; nt < S::NT; ++nt) v[nt] = acc[0][nt][e] + acc[1][nt][e];
      if constexpr (S::NT == 1) l[e] = v[0] + __shfl_xor_sync(0xffffffffu, v[0], 2);
      else l[e] = v[0] + v[1];
    }
    const int k0 = r0 + gid, k1 = k0 + 8;
    const bool v0 = k0 < nrows, v1 = k1 < nrows;
    if (!v0) l[0] = l[1] = -INFINITY;
    if (!v1) l[2] = l[3] = -INFINITY;
    float* lg = a.logits + ((size_t)seg * a.lstride + row0) * G;   // [position][G]
    if (hA < G) {
      if constexpr (G == 1) {
        if (v0) lg[k0] = l[0];
        if (v1) lg[k1] = l[2];
      } else {
        if (v0) *reinterpret_cast<float2*>(lg + (size_t)k0 * G + hA) = make_float2(l[0], l[1]);
        if (v1) *reinterpret_cast<float2*>(lg + (size_t)k1 * G + hA) = make_float2(l[2], l[3]);
      }
    }
    // per-head (max, sum 2^(l - max)) over this warp's 16 keys
    float mA = fmaxf(l[0], l[2]), mB = fmaxf(l[1], l[3]);
#pragma unroll
    for (int o = 4; o <= 16; o <<= 1) {
      mA = fmaxf(mA, __shfl_xor_sync(0xffffffffu, mA, o));
      mB = fmaxf(mB, __shfl_xor_sync(0xffffffffu, mB, o));
    }
    float sA = mA == -INFINITY ? 0.f : exp2f(l[0] - mA) + exp2f(l[2] - mA);
    float sB = mB == -INFINITY ? 0.f : exp2f(l[1] - mB) + exp2f(l[3] - mB);
#pragma unroll
    for (int o = 4; o <= 16; o <<= 1) {
      sA += __shfl_xor_sync(0xffffffffu, sA, o);
      sB += __shfl_xor_sync(0xffffffffu, sB, o);
    }
    if (gid == 0) {
      const size_t pi = (size_t)tile * S::PPT + warp;
      float2* pp = a.part + ((size_t)b * a.n_q + (size_t)g * G) * a.n_parts + pi;
      if (hA < G) pp[(size_t)hA * a.n_parts] = make_float2(mA, sA);
      if (hB < G) pp[(size_t)hB * a.n_parts] = make_float2(mB, sB);
    }
    ++it;
  }
}

// ============================================================== group score + Top-K
// One kernel, one thread-block cluster of C CTAs per (request, KV head); rank
// r owns the contiguous positions [r*slice, (r+1)*slice):
//  * logsumexp of each head of the group over the scan's (max, sum) partials:
//    every rank folds all of them when they are few, else each folds a share
//    and the C results meet through distributed shared memory;
//  * group score s = max_h (l_h - lse_h), p = 2^s (written out on request)
//    and the order key of p (its float bits + 1; 0 marks a forced or absent
//    position), kept in shared memory (global spill for very long slices),
//    with this rank's histogram of the key's bits 30..20;
//  * every rank sums the C histograms and finds the bin that holds the
//    (K - |F|)-th largest key. Usually few keys fall in that bin: every rank
//    then gathers all ranks' keys of the bin and finishes the select on them
//    alone (bits 19..10, then 9..0), and the same gathered keys give each
//    rank its output offset. When the bin holds very many equal-prefix keys
//    the two finer levels are histogrammed over the cluster instead;
//  * an ordered compaction of the rank's slice (ascending positions, keys
//    equal to the threshold to the lowest positions).
constexpr int kSelThreads = 512;
constexpr int kSelMaxCluster = 16;
constexpr int kHistBins = 2048;       // level 1: key bits 30..20
constexpr int kSubBins = 1024;        // levels 2 and 3: bits 19..10, 9..0
constexpr int kSelSmemKeys = 8192;    // keys of a slice kept in shared memory up to this count
constexpr int kSelCandMax = 4096;     // threshold-bin keys finished per rank
constexpr int kSelLseLocal = 8192;    // partials (all heads) a rank folds alone

struct SelArgs {
  const float* logits;
  const float2* part;
  uint32_t* keys;        // global key spill, [segment][kstride]
  int32_t* len;
  float* scores_out;
  int32_t* selected;
  uint32_t* done;
  int B, n_q, n_kv, cap, lstride, K, n_sink, n_recent, append, n_parts, ppt, kstride, C, slice, cpt;
};

struct SelSmem {
  uint32_t hist[kHistBins];           // this rank's histogram of the current level
  uint32_t tot[kHistBins];            // the cluster's counts (or this rank's share of them)
  uint32_t coarse[kHistBins / 32];    // this rank's level-1 counts per 32 bins
  uint32_t keys[kSelSmemKeys];
  uint32_t lc[kSelCandMax];           // this rank's keys in the threshold bin (any order)
  uint32_t cand[kSelCandMax];         // every rank's, in rank order
  float pm[SPC_MAX_GROUP], ps[SPC_MAX_GROUP], lse[SPC_MAX_GROUP];
  float wm[SPC_MAX_GROUP > kSelThreads / 32 ? SPC_MAX_GROUP : kSelThreads / 32];   // per-(head, warp) logsumexp partials
  float ws[SPC_MAX_GROUP > kSelThreads / 32 ? SPC_MAX_GROUP : kSelThreads / 32];
  int scratch[33];
  int cnt[2];                         // published counts of this rank
  int ncand;
  int rb[kSelMaxCluster + 1];         // candidate offsets of the ranks
  int bin, rem, whole;
};

__device__ __forceinline__ bool is_forced(int p, int L, int n_sink, int n_recent) {
  return p < n_sink || p >= L - n_recent;
}

// Bin (scanning from the top) where the running count reaches `rem`, over
// `nbins` counts in shared memory (nbins a multiple of the block size): writes
// the bin, rem minus the count above it, and whether the bin is taken whole.
__device__ __forceinline__ void find_bin(const uint32_t* cnt, int nbins, int rem, SelSmem& sm) {
  const int per = nbins / kSelThreads;
  const int d0 = threadIdx.x * per;   // descending rank of this thread's first bin
  int local = 0;
  for (int j = 0; j < per; ++j) local += (int)cnt[nbins - 1 - (d0 + j)];
  int tot;
  int before = block_excl_scan(local, sm.scratch, &tot);
  for (int j = 0; j < per; ++j) {
    const int bin = nbins - 1 - (d0 + j);
    const int c = (int)cnt[bin];
    if (before < rem && before + c >= rem) {
      sm.bin = bin;
      sm.rem = rem - before;
      sm.whole = (before + c == rem);
    }
    before += c;
  }
  __syncthreads();
}

// Sum over the block of one int per thread (contains __syncthreads).
__device__ __forceinline__ int block_sum(int v, int* scratch) {
  int tot;
  block_excl_scan(v, scratch, &tot);
  return tot;
}

template <int G>
__global__ void __launch_bounds__(kSelThreads) select_kernel(SelArgs a) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ __align__(16) uint8_t sel_smem[];
  SelSmem& sm = *reinterpret_cast<SelSmem*>(sel_smem);
  const int C = a.C;
  const int rank = (int)cluster.block_rank();
  const int seg = blockIdx.x / C;
  const int b = seg / a.n_kv, g = seg - b * a.n_kv;
  const int L = effective_len(a.len, b, a.append, a.cap);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int NW = kSelThreads / 32;
  const bool topk = L > a.K;
  const int Kp = a.K - (a.n_sink + a.n_recent);

  // ---- logsumexp of each head: NW / G warps per head (one when G >= NW),
  // eight partial loads in flight per lane
  const int nv = ((L + kScanRows - 1) / kScanRows) * a.ppt;
  const bool lse_local = (long long)nv * G <= kSelLseLocal;
  {
    constexpr int WPH = G >= NW ? 1 : NW / G;
    const int sub = warp % WPH;
    const int r0 = lse_local ? 0 : (int)((long long)nv * rank / C);
    const int r1 = lse_local ? nv : (int)((long long)nv * (rank + 1) / C);
    const int v0 = r0 + (int)((long long)(r1 - r0) * sub / WPH);
    const int v1 = r0 + (int)((long long)(r1 - r0) * (sub + 1) / WPH);
    for (int h = warp / WPH; h < G; h += NW / WPH) {
      const float2* ph = a.part + ((size_t)b * a.n_q + (size_t)g * G + h) * a.n_parts;
      float m = -INFINITY, s = 0.f;
      for (int i0 = v0 + lane; i0 < v1; i0 += 32 * 8) {
        float2 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = i0 + 32 * u < v1 ? __ldcg(ph + i0 + 32 * u) : make_float2(-INFINITY, 0.f);
#pragma unroll
        for (int u = 0; u < 8; ++u) lse2_combine(m, s, v[u].x, v[u].y);
      }
      warp_lse2(m, s);
      if (lane == 0) { sm.wm[h * WPH + sub] = m; sm.ws[h * WPH + sub] = s; }
    }
  }
  __syncthreads();
  for (int h = tid; h < G; h += kSelThreads) {
    constexpr int WPH = G >= NW ? 1 : NW / G;
    float m = -INFINITY, s = 0.f;
    for (int w = 0; w < WPH; ++w) lse2_combine(m, s, sm.wm[h * WPH + w], sm.ws[h * WPH + w]);
    sm.pm[h] = m;
    sm.ps[h] = s;
    sm.lse[h] = s > 0.f ? m + log2f(s) : INFINITY;
  }
  for (int i = tid; i < kHistBins; i += kSelThreads) sm.hist[i] = 0u;
  if (!lse_local) {
    cluster.sync();
    for (int h = tid; h < G; h += kSelThreads) {
      float rm[kSelMaxCluster], rs[kSelMaxCluster];
#pragma unroll
      for (int r = 0; r < kSelMaxCluster; ++r)
        if (r < C) { rm[r] = *cluster.map_shared_rank(&sm.pm[h], r); rs[r] = *cluster.map_shared_rank(&sm.ps[h], r); }
      float m = -INFINITY, s = 0.f;
#pragma unroll
      for (int r = 0; r < kSelMaxCluster; ++r)
        if (r < C) lse2_combine(m, s, rm[r], rs[r]);
      sm.lse[h] = s > 0.f ? m + log2f(s) : INFINITY;
    }
  }
  __syncthreads();

  // ---- group score, its key, and the level-1 histogram of this rank's slice
  const int p_lo = rank * a.slice;
  const int p_end = min(L, p_lo + a.slice);
  const int t0 = p_lo + tid * a.cpt;
  const int t1 = min(p_end, t0 + a.cpt);
  uint32_t* kb = a.slice <= kSelSmemKeys ? sm.keys : a.keys + (size_t)seg * a.kstride + p_lo;
  // logits are position-major ([position][G]): a group of 4 positions is 4*G
  // consecutive floats, read as G float4 loads. Groups are dealt to threads
  // round robin (a warp reads 32 consecutive groups), every thread runs the
  // same number of rounds, and the histogram increments are aggregated over
  // the lanes of a warp that hit the same bin (the keys of one context crowd
  // into few bins).
  const float* lg = a.logits + (size_t)seg * a.lstride * G;
  constexpr int HC = G < 8 ? G : 8;   // float4 loads in flight together
  const int n_grp = p_end > p_lo ? (p_end - p_lo + 3) >> 2 : 0;
  const int n_rounds = (n_grp + kSelThreads - 1) / kSelThreads;
  // groups of up to 8 heads: the next round's loads are issued before the
  // current ones are used
  constexpr int NPF = G <= 8 ? G : 1;
  float4 pf[NPF];
  if (G <= 8 && tid < n_grp) {
#pragma unroll
    for (int c = 0; c < NPF; ++c) pf[c] = __ldcg(reinterpret_cast<const float4*>(lg + (size_t)(p_lo + 4 * tid) * G) + c);
  }
  for (int rd = 0; rd < n_rounds; ++rd) {
    const int gi = rd * kSelThreads + tid;
    const bool gv = gi < n_grp;
    const int p = p_lo + 4 * gi;
    float sc[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    if (gv) {
      const float4* l4 = reinterpret_cast<const float4*>(lg + (size_t)p * G);
#pragma unroll
      for (int c0 = 0; c0 < G; c0 += HC) {
        float4 v[HC];
        if constexpr (G <= 8) {
#pragma unroll
          for (int c = 0; c < HC; ++c) v[c] = pf[c];
          if (gi + kSelThreads < n_grp) {
#pragma unroll
            for (int c = 0; c < NPF; ++c) pf[c] = __ldcg(l4 + (size_t)kSelThreads * G + c);
          }
        } else {
#pragma unroll
          for (int c = 0; c < HC; ++c) v[c] = __ldcg(l4 + c0 + c);
        }
#pragma unroll
        for (int c = 0; c < HC; ++c) {
          const float f[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int flat = (c0 + c) * 4 + e;      // position p + flat / G, head flat % G
            const int j = flat / G, h = flat - j * G;
            sc[j] = fmaxf(sc[j], f[e] - sm.lse[h]);
          }
        }
      }
    }
    uint32_t key[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int pos = p + j;
      if (gv && pos < p_end) {
        const float pr = exp2f(sc[j]);
        if (a.scores_out) a.scores_out[(size_t)seg * a.cap + pos] = pr;
        key[j] = is_forced(pos, L, a.n_sink, a.n_recent) ? 0u : __float_as_uint(pr) + 1u;
      }
      if (topk) {
        const uint32_t bin = key[j] ? key[j] >> 20 : 0xffffffffu;
        if (n_rounds > 1) {   // long slices: aggregate equal bins over the warp first
          const uint32_t peers = __match_any_sync(0xffffffffu, bin);
          if (bin != 0xffffffffu && lane == __ffs(peers) - 1) atomicAdd(&sm.hist[bin], (uint32_t)__popc(peers));
        } else if (bin != 0xffffffffu) {
          atomicAdd(&sm.hist[bin], 1u);
        }
      }
    }
    // positions past the end keep key 0: the 4-key groups below read them
    if (gv) *reinterpret_cast<uint4*>(kb + (p - p_lo)) = make_uint4(key[0], key[1], key[2], key[3]);
  }
  __syncthreads();   // the passes below read keys other threads wrote

  int32_t* out = a.selected + (size_t)seg * a.K;
  if (!topk) {
    // select all: positions 0..L-1, then -1
    const int i0 = (int)((long long)a.K * rank / C), i1 = (int)((long long)a.K * (rank + 1) / C);
    for (int i = i0 + tid; i < i1; i += kSelThreads) out[i] = i < L ? i : -1;
  } else {
  // ---- threshold key T: the Kp-th largest non-forced key; `need` keys equal
  // to T are taken (T = all-ones and need = 0 when nothing but F is taken).
  // base_b / base_e: selected keys above T / equal to T in lower ranks.
  uint32_t T = 0xffffffffu;
  int need = 0;
  int base_b = -1, base_e = 0;        // base_b < 0: offsets still to exchange
  if (Kp > 0) {
    // the threshold bin in two levels: this rank's counts per 32 bins first,
    // then (one warp) the cluster's sums of those 64 coarse counts and of the
    // 32 bins of the coarse bin that holds the Kp-th key; each rank reads
    // 1 536 remote counts instead of all 2 048 bins of every rank
    for (int j = warp; j < kHistBins / 32; j += NW) {
      const uint32_t v = __reduce_add_sync(0xffffffffu, sm.hist[j * 32 + lane]);
      if (lane == 0) sm.coarse[j] = v;
    }
    cluster.sync();                   // every rank's level-1 histograms are final
    if (warp == 0) {
      const uint32_t kp = (uint32_t)Kp;
      // coarse bins from the top: lane l takes 63 - 2l and 62 - 2l
      const int ja = kHistBins / 32 - 1 - 2 * lane, jb = ja - 1;
      uint32_t va[kSelMaxCluster], vb[kSelMaxCluster];
#pragma unroll
      for (int r = 0; r < kSelMaxCluster; ++r) {
        va[r] = r < C ? *cluster.map_shared_rank(&sm.coarse[ja], r) : 0u;
        vb[r] = r < C ? *cluster.map_shared_rank(&sm.coarse[jb], r) : 0u;
      }
      uint32_t c0 = 0u, c1 = 0u;
#pragma unroll
      for (int r = 0; r < kSelMaxCluster; ++r) { c0 += va[r]; c1 += vb[r]; }
      uint32_t incl = c0 + c1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      const uint32_t before = incl - (c0 + c1);
      int J = -1;
      uint32_t remJ = 0u;
      if (before < kp && kp <= before + c0) { J = ja; remJ = kp - before; }
      else if (before + c0 < kp && kp <= before + c0 + c1) { J = jb; remJ = kp - before - c0; }
      const uint32_t found = __ballot_sync(0xffffffffu, J >= 0);
      const int src = found ? __ffs(found) - 1 : 0;
      J = __shfl_sync(0xffffffffu, J, src);
      remJ = __shfl_sync(0xffffffffu, remJ, src);
      if (J < 0) J = 0;
      // the 32 bins of coarse bin J from the top: lane k takes bin 32 J + 31 - k
      const int bi = J * 32 + 31 - lane;
      uint32_t vf[kSelMaxCluster];
#pragma unroll
      for (int r = 0; r < kSelMaxCluster; ++r) vf[r] = r < C ? *cluster.map_shared_rank(&sm.hist[bi], r) : 0u;
      uint32_t fc = 0u;
#pragma unroll
      for (int r = 0; r < kSelMaxCluster; ++r) fc += vf[r];
      sm.tot[bi] = fc;
      uint32_t fin = fc;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, fin, o);
        if (lane >= o) fin += t;
      }
      const uint32_t fb = fin - fc;
      if (fb < remJ && remJ <= fb + fc) {
        sm.bin = bi;
        sm.rem = (int)(remJ - fb);
        sm.whole = (fb + fc == remJ);
      }
    }
    __syncthreads();
    const uint32_t b1 = (uint32_t)sm.bin;
    const int rem1 = sm.rem;
    if (sm.whole) {
      T = b1 ? (b1 << 20) - 1u : 0u;
    } else if ((int)sm.tot[b1] <= kSelCandMax) {
      // this rank's keys in bin b1, and its count of forced + above-bin keys
      if (tid == 0) sm.ncand = 0;
      __syncthreads();
      int above = 0;
      for (int p = t0; p < t1; ++p) {
        const uint32_t k = kb[p - p_lo];
        if (is_forced(p, L, a.n_sink, a.n_recent) || (k >> 20) > b1) ++above;
        else if (k && (k >> 20) == b1) sm.lc[atomicAdd(&sm.ncand, 1)] = k;
      }
      above = block_sum(above, sm.scratch);
      if (tid == 0) sm.cnt[0] = above;
      cluster.sync();                 // candidates and counts of every rank published
      // candidate counts of the ranks (one load each, in parallel), their
      // offsets, then every candidate copied by its own thread
      int nc_r = 0, ab_r = 0;
      if (tid < C) {
        nc_r = *cluster.map_shared_rank(&sm.ncand, tid);
        if (tid < rank) ab_r = *cluster.map_shared_rank(&sm.cnt[0], tid);
      }
      if (tid < C) sm.rb[tid + 1] = nc_r;
      const int ab_lower = block_sum(ab_r, sm.scratch);
      if (tid == 0) {
        sm.rb[0] = 0;
        for (int r = 0; r < C; ++r) sm.rb[r + 1] += sm.rb[r];
      }
      __syncthreads();
      for (int i = tid; i < sm.rb[C]; i += kSelThreads) {
        int r = 0;
        while (sm.rb[r + 1] <= i) ++r;
        sm.cand[i] = *cluster.map_shared_rank(&sm.lc[i - sm.rb[r]], r);
      }
      __syncthreads();
      const int ncand = sm.rb[C];
      // levels 2 and 3 over the gathered keys
      uint32_t prefix = b1 << 20, pmask = 0xfff00000u;
      int rem = rem1;
      for (int lvl = 1; lvl < 3; ++lvl) {
        const int shift = lvl == 1 ? 10 : 0;
        for (int i = tid; i < kSubBins; i += kSelThreads) sm.hist[i] = 0u;
        __syncthreads();
        for (int i = tid; i < ncand; i += kSelThreads) {
          const uint32_t k = sm.cand[i];
          if ((k & pmask) == prefix) atomicAdd(&sm.hist[(k >> shift) & (kSubBins - 1)], 1u);
        }
        __syncthreads();
        find_bin(sm.hist, kSubBins, rem, sm);
        const uint32_t lower = prefix | ((uint32_t)sm.bin << shift);
        if (sm.whole) { T = lower ? lower - 1u : 0u; need = 0; break; }
        if (lvl == 2) { T = lower; need = sm.rem; break; }
        prefix = lower;
        pmask |= (uint32_t)(kSubBins - 1) << shift;
        rem = sm.rem;
        __syncthreads();
      }
      // offsets of this rank: lower ranks' keys above T and equal to T
      int gt = 0, eq = 0;
      for (int i = tid; i < sm.rb[rank]; i += kSelThreads) {
        const uint32_t k = sm.cand[i];
        gt += k > T;
        eq += k == T;
      }
      base_b = ab_lower + block_sum(gt, sm.scratch);
      base_e = need > 0 ? block_sum(eq, sm.scratch) : 0;
    } else {
      // very many keys share the threshold bin's prefix: histogram the two
      // finer levels over the cluster
      uint32_t prefix = b1 << 20, pmask = 0xfff00000u;
      int rem = rem1;
      for (int lvl = 1; lvl < 3; ++lvl) {
        const int shift = lvl == 1 ? 10 : 0;
        cluster.sync();               // no peer still reads this rank's last histogram
        for (int i = tid; i < kSubBins; i += kSelThreads) sm.hist[i] = 0u;
        __syncthreads();
        for (int p = t0; p < t1; ++p) {
          const uint32_t k = kb[p - p_lo];
          if (k && (k & pmask) == prefix) atomicAdd(&sm.hist[(k >> shift) & (kSubBins - 1)], 1u);
        }
        cluster.sync();
        for (int i = tid; i < kSubBins; i += kSelThreads) {
          uint32_t sum = 0u;
          for (int r = 0; r < C; ++r) sum += *cluster.map_shared_rank(&sm.hist[i], r);
          sm.tot[i] = sum;
        }
        __syncthreads();
        find_bin(sm.tot, kSubBins, rem, sm);
        const uint32_t lower = prefix | ((uint32_t)sm.bin << shift);
        if (sm.whole) { T = lower ? lower - 1u : 0u; need = 0; break; }
        if (lvl == 2) { T = lower; need = sm.rem; break; }
        prefix = lower;
        pmask |= (uint32_t)(kSubBins - 1) << shift;
        rem = sm.rem;
      }
    }
  }

  // ---- ordered compaction of this rank's slice: thread t owns the 4-key
  // groups [t0, t1) (one 16-byte read each)
  int nb_ = 0, ne_ = 0;
  for (int p = t0; p < t1; p += 4) {
    const uint4 k4 = *reinterpret_cast<const uint4*>(kb + (p - p_lo));
    const uint32_t kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int q = p + j;
      if (q >= t1) break;
      if (is_forced(q, L, a.n_sink, a.n_recent) || (kk[j] && kk[j] > T)) ++nb_;
      else if (need > 0 && kk[j] && kk[j] == T) ++ne_;
    }
  }
  int tb, te;
  int off_b = block_excl_scan(nb_, sm.scratch, &tb);
  int off_e = block_excl_scan(ne_, sm.scratch, &te);
  if (base_b < 0) {
    // offsets from the lower ranks' published counts
    if (tid == 0) { sm.cnt[0] = tb; sm.cnt[1] = te; }
    cluster.sync();
    base_b = 0;
    base_e = 0;
    for (int r = 0; r < rank; ++r) {
      base_b += *cluster.map_shared_rank(&sm.cnt[0], r);
      base_e += *cluster.map_shared_rank(&sm.cnt[1], r);
    }
  }
  off_b += base_b;
  off_e += base_e;
  int o = off_b + min(off_e, need);
  int eq_seen = off_e;
  for (int p = t0; p < t1; p += 4) {
    const uint4 k4 = *reinterpret_cast<const uint4*>(kb + (p - p_lo));
    const uint32_t kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int q = p + j;
      if (q >= t1) break;
      bool sel = is_forced(q, L, a.n_sink, a.n_recent) || (kk[j] && kk[j] > T);
      if (!sel && need > 0 && kk[j] && kk[j] == T) {
        sel = eq_seen < need;
        ++eq_seen;
      }
      if (sel) {
        if (o < a.K) out[o] = q;
        ++o;
      }
    }
  }
  }  // topk
  // no rank leaves while a peer may still read its shared memory
  cluster.sync();

  if (a.append && rank == 0 && tid == 0) {
    __threadfence();
    if (atomicAdd(a.done, 1u) == gridDim.x / C - 1) {
      __threadfence();
      for (int bb = 0; bb < a.B; ++bb) {
        const int L0 = a.len[bb];
        if (L0 >= 0 && L0 < a.cap) a.len[bb] = L0 + 1;
      }
      *a.done = 0u;
    }
  }
}

// ============================================================== host side
struct ScoreLayout {
  size_t status, done, q, logits, part_scan, lse, part1, keys, total;
  int n_tiles, ppt, n_parts, lstride;
};

// Groups of up to 8 heads: the mma.sync key scan writes base-2 logits
// [B][n_kv][cap][G] and the select folds them. Groups of 16+ heads: the two
// tcgen05 passes of scan_tc.cu (no logits; one log2 group score per position).
static int scan_ppt(int G) { return G <= 8 ? kScanKmWarps : scan_tc_ppt(G); }

static ScoreLayout score_layout(int B, int H, int n_q, int n_kv, int cap) {
  ScoreLayout l{};
  const int Nq = n_q * kD;
  const bool tc = n_q / n_kv >= 16;
  (void)H;
  l.n_tiles = (cap + kScanRows - 1) / kScanRows;
  l.ppt = scan_ppt(n_q / n_kv);
  l.n_parts = l.n_tiles * l.ppt;
  l.lstride = (cap + 3) & ~3;
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = (off + bytes + 255) & ~size_t(255); return o; };
  l.status = take(2 * sizeof(int));
  l.done = l.status + sizeof(int);
  l.q = take(sizeof(float) * (size_t)B * Nq);
  // logits (G <= 8), or the log2 group scores (G >= 16)
  l.logits = take(sizeof(float) * (size_t)B * (tc ? n_kv : n_q) * l.lstride);
  l.part_scan = take(sizeof(float2) * (size_t)B * n_q * l.n_parts);
  l.lse = tc ? take(sizeof(float) * (size_t)B * n_q) : 0;
  l.part1 = tc ? take(sizeof(float2) * (size_t)B * n_kv * l.n_tiles) : 0;
  l.keys = take(sizeof(uint32_t) * (size_t)B * n_kv * ((cap + 3) & ~3));
  l.total = off;
  return l;
}

size_t score_select_workspace(int B, int H, int n_q, int n_kv, int cap) {
  return score_layout(B, H, n_q, n_kv, cap).total;
}

// Groups of up to 8 heads: the key-major mma.sync kernel (larger groups run
// the tcgen05 passes of scan_tc.cu).
template <int G>
static cudaError_t launch_scan(const ScanArgs& sa, int grid, cudaStream_t st) {
  static_assert(G <= 8, "groups of 16+ heads use scan_tc.cu");
  const size_t smem = kScanSmem;
  cudaError_t e = set_func_attr((const void*)scan_kernel_km<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  scan_kernel_km<G><<<grid, kScanKmThreads, smem, st>>>(sa);
  return cudaGetLastError();
}

// Splits per column tile (the cluster size): one per 256 hidden rows, at most
// 16; a size the device cannot co-schedule is halved.
template <int BB>
static int launch_proj(ProjArgs& pa, int n_tiles, int bz, cudaStream_t st) {
  if (set_func_attr((const void*)proj_kernel<BB>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
    return SPC_ERR_CUDA;
  int S = pa.H / 256;
  S = S < 1 ? 1 : (S > kProjMaxSplit ? kProjMaxSplit : S);
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute at[1];
  cfg.blockDim = dim3(kProjThreads, 1, 1);
  cfg.stream = st;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  at[0].id = cudaLaunchAttributeClusterDimension;
  for (;; S /= 2) {
    pa.S = S;
    pa.Hc = (pa.H + S - 1) / S;
    const size_t smem = sizeof(float) * ((size_t)pa.Hc * BB + (kProjThreads / 32) * BB * kProjTile);
    if (set_func_attr((const void*)proj_kernel<BB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return SPC_ERR_CUDA;
    cfg.gridDim = dim3(n_tiles * S, 1, bz);
    cfg.dynamicSmemBytes = smem;
    at[0].val.clusterDim.x = S;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    int n_clusters = 0;
    if (S == 1 || (cudaOccupancyMaxActiveClusters(&n_clusters, proj_kernel<BB>, &cfg) == cudaSuccess &&
                   n_clusters > 0))
      break;
    cudaGetLastError();
  }
  return cudaLaunchKernelEx(&cfg, proj_kernel<BB>, pa) == cudaSuccess ? SPC_OK : SPC_ERR_CUDA;
}

// The tensor-core projection: the splits per column tile (the cluster size)
// are the largest power of two that keeps the grid within one wave of two
// CTAs per SM, at most 16 and at most one per 256 hidden rows, so every CTA
// streams a long run of weight rows; split boundaries fall on multiples of 8
// hidden rows.
static int launch_proj_tc(ProjArgs& pa, int n_tiles, int bz, cudaStream_t st) {
  if (set_func_attr((const void*)proj_tc_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
    return SPC_ERR_CUDA;
  const long long slots = 2LL * (device_sm_count() > 0 ? device_sm_count() : 1);
  int S = 1;
  while (S < kProjMaxSplit && 2 * S * 256 <= pa.H && (long long)n_tiles * bz * 2 * S <= slots) S *= 2;
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute at[1];
  cfg.blockDim = dim3(kPtcThreads, 1, 1);
  cfg.stream = st;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  at[0].id = cudaLaunchAttributeClusterDimension;
  for (;; S /= 2) {
    pa.S = S;
    pa.Hc = ((pa.H + S - 1) / S + 7) / 8 * 8;
    const size_t smem = kPtcSmem;
    if (set_func_attr((const void*)proj_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return SPC_ERR_CUDA;
    cfg.gridDim = dim3(n_tiles * S, 1, bz);
    cfg.dynamicSmemBytes = smem;
    at[0].val.clusterDim.x = S;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    int n_clusters = 0;
    if (S == 1 || (cudaOccupancyMaxActiveClusters(&n_clusters, proj_tc_kernel, &cfg) == cudaSuccess &&
                   n_clusters > 0))
      break;
    cudaGetLastError();
  }
  return cudaLaunchKernelEx(&cfg, proj_tc_kernel, pa) == cudaSuccess ? SPC_OK : SPC_ERR_CUDA;
}

// Cluster size: at most two CTAs per SM over all segments, at most 16, and
// at least 512 positions per CTA; a size the device cannot co-schedule is
// halved.
template <int G>
static int launch_select(SelArgs& sa, int nseg, cudaStream_t st) {
  const size_t smem = sizeof(SelSmem);
  if (set_func_attr((const void*)select_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
          cudaSuccess ||
      set_func_attr((const void*)select_kernel<G>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
    return SPC_ERR_CUDA;
  int C = 1;
  while (C < kSelMaxCluster && nseg * C * 2 <= 2 * device_sm_count() && sa.cap / (C * 2) >= 512) C *= 2;
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute at[1];
  cfg.blockDim = dim3(kSelThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  at[0].id = cudaLaunchAttributeClusterDimension;
  for (;; C /= 2) {
    cfg.gridDim = dim3(nseg * C, 1, 1);
    at[0].val.clusterDim.x = C;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    int n_clusters = 0;
    if (C == 1 || (cudaOccupancyMaxActiveClusters(&n_clusters, select_kernel<G>, &cfg) == cudaSuccess &&
                   n_clusters > 0))
      break;
    cudaGetLastError();
  }
  const int per_rank = (sa.cap + C - 1) / C;
  sa.C = C;
  sa.cpt = (((per_rank + kSelThreads - 1) / kSelThreads) + 3) & ~3;
  sa.slice = (per_rank + 3) & ~3;
  if (cudaLaunchKernelEx(&cfg, select_kernel<G>, sa) != cudaSuccess) return SPC_ERR_CUDA;
  return SPC_OK;
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
    pa.status = status;
    pa.B = c.B; pa.H = c.H; pa.Nq = Nq; pa.Nk = Nk; pa.Ntot = Nq + Nk; pa.n_kv = c.n_kv;
    pa.cap = c.cap;
    const int n_tiles = (Nq + (c.append ? Nk : 0)) / kProjTile;
    const int bb = c.B <= 1 ? 1 : c.B <= 2 ? 2 : c.B <= 4 ? 4 : c.B <= 8 ? 8 : 16;
    const int bz = (c.B + bb - 1) / bb;
    int rc;
    if (c.B >= SPC_PROJ_TC_MIN_BATCH) {
      rc = launch_proj_tc(pa, n_tiles, (c.B + 15) / 16, st);
      if (rc != SPC_OK) return rc;
    } else switch (bb) {
      case 1: rc = launch_proj<1>(pa, n_tiles, bz, st); break;
      case 2: rc = launch_proj<2>(pa, n_tiles, bz, st); break;
      case 4: rc = launch_proj<4>(pa, n_tiles, bz, st); break;
      case 8: rc = launch_proj<8>(pa, n_tiles, bz, st); break;
      default: rc = launch_proj<16>(pa, n_tiles, bz, st); break;
    }
    if (rc != SPC_OK) return rc;
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
    sa.n_q = c.n_q; sa.n_kv = c.n_kv; sa.cap = c.cap; sa.lstride = l.lstride; sa.n_tiles = l.n_tiles;
    sa.total_tiles = c.B * c.n_kv * l.n_tiles; sa.append = c.append; sa.n_parts = l.n_parts;
    sa.qscale = kLog2e / sqrtf((float)kD);
    if (G >= 16) {
      ScanTcCall tc{};
      tc.K = sa.K; tc.q = sa.q; tc.len = sa.len; tc.part = sa.part; tc.status = status;
      tc.B = c.B; tc.n_q = c.n_q; tc.n_kv = c.n_kv; tc.cap = c.cap; tc.lstride = l.lstride;
      tc.n_tiles = l.n_tiles; tc.total_tiles = sa.total_tiles; tc.append = c.append; tc.n_parts = l.n_parts;
      tc.qscale = sa.qscale;
      const int rc = scan_tc_launch(tc, G, c.stream);
      if (rc != SPC_OK) return rc;
    } else {
      // each CTA takes a run of consecutive tiles
      if (kScanTilesPerCta > 0) {
        sa.tpc = kScanTilesPerCta;
      } else {
        const long long slots = (long long)kScanCtasPerSm * (device_sm_count() > 0 ? device_sm_count() : 1);
        sa.tpc = (int)((sa.total_tiles + slots - 1) / slots);
        if (sa.tpc < 1) sa.tpc = 1;
      }
      const int grid = (sa.total_tiles + sa.tpc - 1) / sa.tpc;
      switch (G) {
        case 1: e = launch_scan<1>(sa, grid, st); break;
        case 2: e = launch_scan<2>(sa, grid, st); break;
        case 4: e = launch_scan<4>(sa, grid, st); break;
        default: e = launch_scan<8>(sa, grid, st); break;
      }
      if (e != cudaSuccess) return SPC_ERR_CUDA;
    }
  }

  // ---- logsumexp, group score, Top-K (one cluster per request and KV head)
  if (c.stages & SPC_STAGE_SELECT) {
    SelArgs sa{};
    sa.logits = reinterpret_cast<const float*>(ws + l.logits);
    sa.part = reinterpret_cast<const float2*>(ws + l.part_scan);
    sa.keys = reinterpret_cast<uint32_t*>(ws + l.keys);
    sa.len = c.len;
    sa.scores_out = c.scores_out;
    sa.selected = c.selected;
    sa.done = reinterpret_cast<uint32_t*>(ws + l.done);
    sa.B = c.B; sa.n_q = c.n_q; sa.n_kv = c.n_kv; sa.cap = c.cap; sa.lstride = l.lstride; sa.K = c.budget;
    sa.n_sink = c.n_sink; sa.n_recent = c.n_recent; sa.append = c.append;
    sa.n_parts = l.n_parts; sa.ppt = l.ppt; sa.kstride = (c.cap + 3) & ~3;
    int rc;
    if (G >= 16) {
      // normalisers, then the second pass over the keys writes one log2 group
      // score per position; the select ranks them as a group of one head
      // with a zero normaliser
      ScanTcCall tc{};
      tc.K = static_cast<const uint16_t*>(c.K_dlm);
      tc.q = reinterpret_cast<const float*>(ws + l.q);
      tc.len = c.len;
      tc.part = reinterpret_cast<float2*>(ws + l.part_scan);
      tc.lse = reinterpret_cast<float*>(ws + l.lse);
      tc.gscore = reinterpret_cast<float*>(ws + l.logits);
      tc.status = status;
      tc.B = c.B; tc.n_q = c.n_q; tc.n_kv = c.n_kv; tc.cap = c.cap; tc.lstride = l.lstride;
      tc.n_tiles = l.n_tiles; tc.total_tiles = c.B * c.n_kv * l.n_tiles; tc.append = c.append;
      tc.n_parts = l.n_parts; tc.qscale = kLog2e / sqrtf((float)kD);
      float2* part1 = reinterpret_cast<float2*>(ws + l.part1);
      rc = scan_tc_scores_launch(tc, G, part1, l.n_tiles, c.stream);
      if (rc != SPC_OK) return rc;
      sa.part = part1;
      sa.n_q = c.n_kv;
      sa.n_parts = l.n_tiles;
      sa.ppt = 1;
      rc = launch_select<1>(sa, c.B * c.n_kv, st);
    } else {
      switch (G) {
        case 1: rc = launch_select<1>(sa, c.B * c.n_kv, st); break;
        case 2: rc = launch_select<2>(sa, c.B * c.n_kv, st); break;
        case 4: rc = launch_select<4>(sa, c.B * c.n_kv, st); break;
        default: rc = launch_select<8>(sa, c.B * c.n_kv, st); break;
      }
    }
    if (rc != SPC_OK) return rc;
  }
  return SPC_OK;
}


// ============================================================== MLA retrieval head
// "ASPLOS'26 | SpeContext ..." (marsggbo blog) §5 and "SpeContext: ..."
// (paperlayer.ai summary) §4.3: with MLA the head scores the latent cache,
// head-level; the latent row is shared by all query heads, so (as for MQA)
// the 16 heads form one group and each request gets one selection.
//
// Latent scan: logits l[b, p, h] = qa[b, h] . C[b, p] * log2(e) / sqrt(192)
// for the absorbed queries qa (576 values: W_uk[h]^T q_nope ; q_rope) over
// the 576-value latent rows. One CTA per SM: a producer warp streams 32-row
// tiles into a 4-stage ring, one bulk copy (cp.async.bulk) per row at a
// 1168-byte pitch (16 bytes of padding keep ldmatrix conflict-free), for
// four consumer warps (a second group of four would
// leave each warp 168 registers, and the query fragments alone take 72).
// The four warps split the 576 dims (9 k-steps of mma.sync
// m16n8k16 each, the 16 heads on the M side, the query in bf16 high and low
// parts so the logits keep fp32 accuracy), sum their partial tiles through
// shared memory, and each finishes 8 of the 32 rows: logits out, one
// logsumexp partial per head per 8 rows (16 per 128 positions).
constexpr int kMsLat = SPC_MLA_LATENT + SPC_MLA_ROPE;   // 576
constexpr int kMsLatBytes = kMsLat * 2;
constexpr int kMsH = SPC_MLA_HEADS;                     // 16
constexpr int kMsQk = SPC_MLA_NOPE + SPC_MLA_ROPE;      // 192
constexpr int kMsRows = 32;
constexpr int kMsStages = 4;
constexpr int kMsGroups = 1;   // nine warps would cap registers at 168 (16K per SM sub-partition)
constexpr int kMsKw = 4;
constexpr int kMsThreads = (kMsGroups * kMsKw + 1) * 32;
constexpr int kMsKs = kMsLat / 16 / kMsKw;              // 9
constexpr int kMsPitch = kMsLatBytes + 16;              // 1168: conflict-free ldmatrix over 8 rows
constexpr uint32_t kMsTile = kMsRows * kMsPitch;        // 36.5 KiB
constexpr int kMsPpt = (kScanRows / kMsRows) * kMsKw;   // 16 partials per 128 positions
constexpr size_t kMsRed = (size_t)kMsGroups * kMsKw * 4 * 32 * 16;
constexpr size_t kMsSmem = kMsStages * (size_t)kMsTile + kMsRed + 2 * kMsStages * sizeof(uint64_t);

struct MlaScanArgs {
  const uint16_t* C;
  const float* qa;
  const int32_t* len;
  float* logits;
  float2* part;
  int* status;
  int cap, lstride, n_tiles, total_tiles, append, n_parts, tpc;
  float qscale;
};

__device__ __forceinline__ void ms_bar(int grp) {
  asm volatile("bar.sync %0, %1;" :: "r"(1 + grp), "n"(kMsKw * 32) : "memory");
}

__global__ void __launch_bounds__(kMsThreads, 1) mla_scan_kernel(MlaScanArgs a) {
  extern __shared__ __align__(128) uint8_t mss[];
  float4* red = reinterpret_cast<float4*>(mss + kMsStages * (size_t)kMsTile);
  uint64_t* full = reinterpret_cast<uint64_t*>(mss + kMsStages * (size_t)kMsTile + kMsRed);
  uint64_t* empty = full + kMsStages;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kMsStages; ++s) {
      mbar_init(&full[s], 1);        // lane 0, 32 row copies expected
      mbar_init(&empty[s], kMsKw);   // the group that owns the stage
    }
    fence_mbar_init();
  }
  __syncthreads();
  const int t_begin = blockIdx.x * a.tpc, t_end = min(a.total_tiles, t_begin + a.tpc);

  if (warp == kMsGroups * kMsKw) {
    // ---------------- producer
    int it = 0;
    for (int t = t_begin; t < t_end; ++t) {
      const int b = t / a.n_tiles, tile = t - b * a.n_tiles;
      const int L = effective_len(a.len, b, a.append, a.cap);
      const int row0 = tile * kMsRows;
      if (row0 >= L) continue;
      const int nrows = min(kMsRows, L - row0);
      const int s = it % kMsStages;
      const uint32_t ph = (it / kMsStages) & 1;
      if (!mbar_wait_bounded(&empty[s], ph ^ 1, kWaitLimit)) {
        if (lane == 0) set_status(a.status, SPC_ERR_TIMEOUT);
        break;
      }
      // one bulk copy per row (lane r: row r); rows past the end copy the
      // tile's first row again (their logits are never written or summed)
      if (lane == 0) mbar_arrive_expect_tx(&full[s], kMsRows * kMsLatBytes);
      __syncwarp();
      bulk_g2s(mss + (size_t)s * kMsTile + lane * kMsPitch,
               a.C + ((size_t)b * a.cap + row0 + (lane < nrows ? lane : 0)) * kMsLat, kMsLatBytes, &full[s]);
      ++it;
    }
    for (int k = max(0, it - kMsStages); k < it; ++k)
      mbar_wait_bounded(&full[k % kMsStages], (k / kMsStages) & 1, kWaitLimit);
    return;
  }

  // ---------------- consumers
  const int grp = warp / kMsKw, kw = warp - grp * kMsKw;
  const int gid = lane >> 2, tig = lane & 3, lm = lane >> 3, lr = lane & 7;
  const uint32_t smem0 = smem_u32(mss);
  float4* rg = red + (size_t)grp * kMsKw * 4 * 32;
  uint32_t qh[kMsKs][4], ql[kMsKs][4];
  int cur_b = -1;
  bool dead = false;
  int it = 0;
  for (int t = t_begin; t < t_end; ++t) {
    const int b = t / a.n_tiles, tile = t - b * a.n_tiles;
    const int L = effective_len(a.len, b, a.append, a.cap);
    const int row0 = tile * kMsRows;
    if (row0 >= L) {
      // a tile past the end inside the last 128-position tile still owes
      // its (empty) logsumexp partials
      if (grp == 0 && (row0 & ~(kScanRows - 1)) < L && lane < kMsH)
        a.part[((size_t)b * kMsH + lane) * a.n_parts + (size_t)tile * kMsKw + kw] = make_float2(-INFINITY, 0.f);
      continue;
    }
    const int my = it++;
    if (my % kMsGroups != grp) continue;
    const int s = my % kMsStages;
    const uint32_t ph = (my / kMsStages) & 1;
    const int nrows = min(kMsRows, L - row0);
    if (b != cur_b) {
      const float* qp = a.qa + (size_t)b * kMsH * kMsLat;
#pragma unroll
      for (int ks = 0; ks < kMsKs; ++ks) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int h = gid + ((e & 1) ? 8 : 0);
          const int c = (kw * kMsKs + ks) * 16 + tig * 2 + ((e & 2) ? 8 : 0);
          const float2 v = *reinterpret_cast<const float2*>(qp + (size_t)h * kMsLat + c);
          const float x = v.x * a.qscale, y = v.y * a.qscale;
          const float xh = bf16_round(x), yh = bf16_round(y);
          qh[ks][e] = pack_bf16(xh, yh);
          ql[ks][e] = pack_bf16(x - xh, y - yh);
        }
      }
      cur_b = b;
    }
    if (!dead && !mbar_wait_bounded(&full[s], ph, kWaitLimit)) {
      if (lane == 0) set_status(a.status, SPC_ERR_TIMEOUT);
      dead = true;
    }
    const uint32_t tb = smem0 + (uint32_t)(s * kMsTile);
    float acc[4][4], acl[4][4];
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[n][e] = acl[n][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < kMsKs; ++ks) {
      const int kg = kw * kMsKs + ks;
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        const int row = np * 16 + ((lm >> 1) << 3) + lr;
        uint32_t b0, b1, b2, b3;
        ldsm_x4(tb + row * kMsPitch + ((kg * 2 + (lm & 1)) << 4), b0, b1, b2, b3);
        mma_bf16(acc[2 * np], qh[ks], b0, b1);
        mma_bf16(acl[2 * np], ql[ks], b0, b1);
        mma_bf16(acc[2 * np + 1], qh[ks], b2, b3);
        mma_bf16(acl[2 * np + 1], ql[ks], b2, b3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
#pragma unroll
    for (int n = 0; n < 4; ++n)
      rg[(kw * 4 + n) * 32 + lane] =
          make_float4(acc[n][0] + acl[n][0], acc[n][1] + acl[n][1], acc[n][2] + acl[n][2], acc[n][3] + acl[n][3]);
    ms_bar(grp);
    float4 v = rg[kw * 32 + lane];
#pragma unroll
    for (int w = 1; w < kMsKw; ++w) {
      const float4 u = rg[(w * 4 + kw) * 32 + lane];
      v.x += u.x; v.y += u.y; v.z += u.z; v.w += u.w;
    }
    ms_bar(grp);
    // rows kw*8 + 2 tig, +1 of the tile; heads gid (x, y) and gid + 8 (z, w)
    const int key = kw * 8 + tig * 2;
    const bool v0 = key < nrows, v1 = key + 1 < nrows;
    float* lg = a.logits + ((size_t)b * a.lstride + row0) * kMsH;
    if (v0) { lg[key * kMsH + gid] = v.x; lg[key * kMsH + gid + 8] = v.z; }
    if (v1) { lg[(key + 1) * kMsH + gid] = v.y; lg[(key + 1) * kMsH + gid + 8] = v.w; }
    if (!v0) v.x = v.z = -INFINITY;
    if (!v1) v.y = v.w = -INFINITY;
    float m_lo = fmaxf(v.x, v.y), m_hi = fmaxf(v.z, v.w);
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      m_lo = fmaxf(m_lo, __shfl_xor_sync(0xffffffffu, m_lo, o));
      m_hi = fmaxf(m_hi, __shfl_xor_sync(0xffffffffu, m_hi, o));
    }
    float s_lo = m_lo == -INFINITY ? 0.f : exp2f(v.x - m_lo) + exp2f(v.y - m_lo);
    float s_hi = m_hi == -INFINITY ? 0.f : exp2f(v.z - m_hi) + exp2f(v.w - m_hi);
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      s_lo += __shfl_xor_sync(0xffffffffu, s_lo, o);
      s_hi += __shfl_xor_sync(0xffffffffu, s_hi, o);
    }
    if (tig == 0) {
      const size_t pi = (size_t)tile * kMsKw + kw;
      a.part[((size_t)b * kMsH + gid) * a.n_parts + pi] = make_float2(m_lo, s_lo);
      a.part[((size_t)b * kMsH + gid + 8) * a.n_parts + pi] = make_float2(m_hi, s_hi);
    }
  }
}

struct MlaLayout {
  size_t status, done, q, qa, logits, part, keys, total;
  int n_tiles, n_parts, lstride;
};

static MlaLayout mla_layout(int B, int cap) {
  MlaLayout l{};
  l.n_tiles = (cap + kMsRows - 1) / kMsRows;
  l.n_parts = ((cap + kScanRows - 1) / kScanRows) * kMsPpt;
  l.lstride = (cap + 3) & ~3;
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = (off + bytes + 255) & ~size_t(255); return o; };
  l.status = take(2 * sizeof(int));
  l.done = l.status + sizeof(int);
  l.q = take(sizeof(float) * (size_t)B * kMsH * kMsQk);
  l.qa = take(sizeof(float) * (size_t)B * kMsH * kMsLat);
  l.logits = take(sizeof(float) * (size_t)B * kMsH * l.lstride);
  l.part = take(sizeof(float2) * (size_t)B * kMsH * l.n_parts);
  l.keys = take(sizeof(uint32_t) * (size_t)B * ((cap + 3) & ~3));
  l.total = off;
  return l;
}

size_t mla_score_select_workspace(int B, int cap) { return mla_layout(B, cap).total; }

int mla_score_select_launch(const MlaScoreSelectCall& c) {
  const MlaLayout l = mla_layout(c.B, c.cap);
  uint8_t* ws = static_cast<uint8_t*>(c.workspace);
  cudaStream_t st = static_cast<cudaStream_t>(c.stream);
  int* status = reinterpret_cast<int*>(ws + l.status);
  float* qws = reinterpret_cast<float*>(ws + l.q);
  float* qa = reinterpret_cast<float*>(ws + l.qa);

  // ---- projection (CUDA cores; the latent row's last tile is partial), absorption
  if (c.stages & SPC_STAGE_PROJECT) {
    ProjArgs pa{};
    pa.x = static_cast<const uint16_t*>(c.x);
    pa.Wq = static_cast<const uint16_t*>(c.Wq);
    pa.Wk = static_cast<const uint16_t*>(c.Wdkv);
    pa.K_dlm = static_cast<uint16_t*>(c.C_dlm);
    pa.len = c.len;
    pa.q_ws = qws;
    pa.q_out = nullptr;
    pa.status = status;
    pa.B = c.B; pa.H = c.H; pa.Nq = kMsH * kMsQk; pa.Nk = kMsLat; pa.Ntot = pa.Nq + pa.Nk; pa.n_kv = 1;
    pa.cap = c.cap; pa.latent = 1;
    const int n_tiles = (pa.Nq + (c.append ? pa.Nk : 0) + kProjTile - 1) / kProjTile;
    const int bb = c.B <= 1 ? 1 : c.B <= 2 ? 2 : c.B <= 4 ? 4 : c.B <= 8 ? 8 : 16;
    const int bz = (c.B + bb - 1) / bb;
    int rc;
    switch (bb) {
      case 1: rc = launch_proj<1>(pa, n_tiles, bz, st); break;
      case 2: rc = launch_proj<2>(pa, n_tiles, bz, st); break;
      case 4: rc = launch_proj<4>(pa, n_tiles, bz, st); break;
      case 8: rc = launch_proj<8>(pa, n_tiles, bz, st); break;
      default: rc = launch_proj<16>(pa, n_tiles, bz, st); break;
    }
    if (rc != SPC_OK) return rc;
    rc = mla_absorb_launch(qws, 0, c.Wuk, c.B, c.B, qa, c.stream);
    if (rc != SPC_OK) return rc;
  }

  // ---- latent scan
  if (c.stages & SPC_STAGE_SCAN) {
    MlaScanArgs sa{};
    sa.C = static_cast<const uint16_t*>(c.C_dlm);
    sa.qa = qa;
    sa.len = c.len;
    sa.logits = reinterpret_cast<float*>(ws + l.logits);
    sa.part = reinterpret_cast<float2*>(ws + l.part);
    sa.status = status;
    sa.cap = c.cap; sa.lstride = l.lstride; sa.n_tiles = l.n_tiles; sa.total_tiles = c.B * l.n_tiles;
    sa.append = c.append; sa.n_parts = l.n_parts;
    sa.qscale = kLog2e / sqrtf((float)kMsQk);
    const int sms = device_sm_count() > 0 ? device_sm_count() : 1;
    sa.tpc = (sa.total_tiles + sms - 1) / sms;
    if (sa.tpc < 1) sa.tpc = 1;
    const int grid = (sa.total_tiles + sa.tpc - 1) / sa.tpc;
    if (set_func_attr((const void*)mla_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMsSmem) !=
        cudaSuccess)
      return SPC_ERR_CUDA;
    mla_scan_kernel<<<grid, kMsThreads, kMsSmem, st>>>(sa);
    if (cudaGetLastError() != cudaSuccess) return SPC_ERR_CUDA;
  }

  // ---- logsumexp, group score over all 16 heads, Top-K (one per request)
  if (c.stages & SPC_STAGE_SELECT) {
    SelArgs sa{};
    sa.logits = reinterpret_cast<const float*>(ws + l.logits);
    sa.part = reinterpret_cast<const float2*>(ws + l.part);
    sa.keys = reinterpret_cast<uint32_t*>(ws + l.keys);
    sa.len = c.len;
    sa.scores_out = c.scores_out;
    sa.selected = c.selected;
    sa.done = reinterpret_cast<uint32_t*>(ws + l.done);
    sa.B = c.B; sa.n_q = kMsH; sa.n_kv = 1; sa.cap = c.cap; sa.lstride = l.lstride; sa.K = c.budget;
    sa.n_sink = c.n_sink; sa.n_recent = c.n_recent; sa.append = c.append;
    sa.n_parts = l.n_parts; sa.ppt = kMsPpt; sa.kstride = (c.cap + 3) & ~3;
    const int rc = launch_select<kMsH>(sa, c.B, st);
    if (rc != SPC_OK) return rc;
  }
  return SPC_OK;
}


// ============================================================== batch-level selection
// "ASPLOS'26 | SpeContext ..." (marsggbo blog) §5 compares head-level
// retrieval with a batch-level one that merges every head's weights into one
// Top-K. Here: per request, the element-wise max over all groups' scores (the
// group probabilities spc_score_select writes to scores_out) is written as a
// base-2 logit with a zero log-normaliser, and the head-level select kernel
// (one group of one head per request) takes the Top-K; the selection is then
// copied to every KV head.
struct BatchLayout {
  size_t status, done, logits, part, keys, sel, total;
  int lstride, n_parts;
};

static BatchLayout batch_layout(int B, int cap, int budget) {
  BatchLayout l{};
  l.lstride = (cap + 3) & ~3;
  l.n_parts = (cap + kScanRows - 1) / kScanRows;
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = (off + bytes + 255) & ~size_t(255); return o; };
  l.status = take(2 * sizeof(int));
  l.done = l.status + sizeof(int);
  l.logits = take(sizeof(float) * (size_t)B * l.lstride);
  l.part = take(sizeof(float2) * (size_t)B * l.n_parts);
  l.keys = take(sizeof(uint32_t) * (size_t)B * l.lstride);
  l.sel = take(sizeof(int32_t) * (size_t)B * budget);
  l.total = off;
  return l;
}

size_t batch_select_workspace(int B, int cap, int budget) { return batch_layout(B, cap, budget).total; }

constexpr int kBcThreads = 256;

__global__ void __launch_bounds__(kBcThreads)
batch_combine_kernel(const float* __restrict__ scores, const int32_t* __restrict__ len, int n_kv, int cap,
                     int lstride, int n_parts, float* __restrict__ logits, float2* __restrict__ part) {
  const int b = blockIdx.y, p = blockIdx.x * kBcThreads + threadIdx.x;
  int L = len[b];
  L = L < 0 ? 0 : (L > cap ? cap : L);
  if (p < L) {
    float m = 0.f;
    for (int g = 0; g < n_kv; ++g) m = fmaxf(m, scores[((size_t)b * n_kv + g) * cap + p]);
    logits[(size_t)b * lstride + p] = m > 0.f ? log2f(m) : -INFINITY;
  }
  // one logsumexp partial per 128 positions: the first is (0, 1), so the
  // select's normaliser is 0 and its probabilities are the merged scores
  if (p < n_parts) part[(size_t)b * n_parts + p] = p == 0 ? make_float2(0.f, 1.f) : make_float2(-INFINITY, 0.f);
}

__global__ void __launch_bounds__(kBcThreads)
batch_broadcast_kernel(const int32_t* __restrict__ sel, int n_kv, int K, long long total, int32_t* __restrict__ out) {
  for (long long i = (long long)blockIdx.x * kBcThreads + threadIdx.x; i < total; i += (long long)gridDim.x * kBcThreads) {
    const long long k = i % K, bg = i / K, b = bg / n_kv;
    out[i] = sel[b * K + k];
  }
}

int batch_select_launch(const float* scores, int32_t* len, int B, int n_kv, int cap, int budget, int n_sink,
                        int n_recent, int32_t* selected, void* workspace, void* stream) {
  const BatchLayout l = batch_layout(B, cap, budget);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int n_blk = (std::max(cap, l.n_parts) + kBcThreads - 1) / kBcThreads;
  batch_combine_kernel<<<dim3(n_blk, B), kBcThreads, 0, st>>>(scores, len, n_kv, cap, l.lstride, l.n_parts,
                                                              reinterpret_cast<float*>(ws + l.logits),
                                                              reinterpret_cast<float2*>(ws + l.part));
  if (cudaGetLastError() != cudaSuccess) return SPC_ERR_CUDA;
  SelArgs sa{};
  sa.logits = reinterpret_cast<const float*>(ws + l.logits);
  sa.part = reinterpret_cast<const float2*>(ws + l.part);
  sa.keys = reinterpret_cast<uint32_t*>(ws + l.keys);
  sa.len = len;
  sa.scores_out = nullptr;
  sa.selected = reinterpret_cast<int32_t*>(ws + l.sel);
  sa.done = reinterpret_cast<uint32_t*>(ws + l.done);
  sa.B = B; sa.n_q = 1; sa.n_kv = 1; sa.cap = cap; sa.lstride = l.lstride; sa.K = budget;
  sa.n_sink = n_sink; sa.n_recent = n_recent; sa.append = 0;
  sa.n_parts = l.n_parts; sa.ppt = 1; sa.kstride = l.lstride;
  const int rc = launch_select<1>(sa, B, st);
  if (rc != SPC_OK) return rc;
  const long long total = (long long)B * n_kv * budget;
  long long grid = (total + kBcThreads - 1) / kBcThreads;
  if (grid > 1024) grid = 1024;
  batch_broadcast_kernel<<<(int)grid, kBcThreads, 0, st>>>(reinterpret_cast<const int32_t*>(ws + l.sel), n_kv,
                                                          budget, total, selected);
  return cudaGetLastError() == cudaSuccess ? SPC_OK : SPC_ERR_CUDA;
}

}  // namespace spc
