// Key scan of the retrieval head for large query-head groups (G = 16, 32, 64;
// the MQA shape is G = 64) on the 5th-generation tensor cores.
//
// Method: "ASPLOS'26 | SpeContext 让小模型先圈出重要 KV Cache" (marsggbo blog)
// §2 (attention weights softmax(q K^T / sqrt(d)) of the retrieval head over
// the whole context) and §5 (for GQA/MQA the weights of a group's query heads
// are combined, so every head of the group scores every position of its KV
// head); "SpeContext: Enabling Efficient Long-context Reasoning with
// Speculative Context Sparsity in LLMs" (paperlayer.ai summary) §3.1 (the
// per-step cost is this scan over the context) and §4.3.
//
// Two passes over the key cache (both HBM-bound, neither writes the logits):
//  * pass 1 (SCAN stage) folds every head's logits into logsumexp partials
//    (max, sum 2^(l - max)) per (head, 128-position tile, slice of the tile);
//  * a fold kernel turns them into each head's normaliser lse_h (base 2);
//  * pass 2 (SELECT stage) recomputes the logits and writes one value per
//    position, the log2 of the group score max_h 2^(l_h - lse_h), which the
//    radix select then ranks as a group of one head with a zero normaliser.
// Logits are (q_h . K[p]) * log2(e) / sqrt(d). Reading the keys twice moves
// 2 x 256 B per position, where writing position-major logits for G = 64
// and reading them back in the select would move 256 + 256 + 256 B.
//
// GB300 design, one CTA per SM, warp-specialised:
//  * work split: a CTA takes tiles of one segment (request, KV head) while
//    every segment can have CTAs of its own, the CTAs of a segment
//    interleaved tile by tile (one advancing front per segment reads the
//    cache faster than one run per CTA); each CTA stages its first segment's
//    queries with all its threads before any key copy is issued.
//  * warp 0, one lane: TMA producer. Each 128-position key tile (32 KiB) comes
//    in as two 64-dimension boxes of a 3-D tensor map ([segment][position]
//    [dim]) with the 128-byte swizzle, into a 6-stage ring (192 KiB in flight
//    per SM); completion is counted in bytes on the stage's mbarrier.
//    Positions past the capacity are zero-filled by the copy and masked.
//  * warp 1: allocates the tensor memory (two accumulators), rebuilds the
//    query operand when a run crosses into another segment (the group's
//    queries scaled by log2(e)/sqrt(d), split into a bf16 high part and a
//    bf16 low part so that q.K keeps ~16 significant bits of q), and one lane
//    issues the MMAs, K = 16 per instruction, 8 instructions per tile, both
//    operands K-major with the 128-byte swizzle; tcgen05.commit frees the key
//    stage and publishes the accumulator.
//    Pass 1: D[128 query rows][128 positions] = Q x K_tile^T with head h's
//    high part in row 2h and its low part in row 2h + 1 (the 2G rows repeated
//    64 / G times), so that one thread holds one head over a run of positions
//    and the pair (2h, 2h + 1) adds its parts with one shuffle per value.
//    Pass 2: D[128 positions][2G] = K_tile x Q^T (high parts in columns
//    [0, G), low parts in [G, 2G)), one position per thread.
//  * epilogue warps (CG column groups of 4, CG = 2 for G = 64), warp w on TMEM
//    lanes 32 (w % 4) .. +31 with tcgen05.ld. Pass 1: each thread folds its
//    head over its share of the positions into one (max, sum) partial;
//    pass 2: the maximum over the thread's heads of l_h - lse_h, the column
//    groups combined through shared memory, 128 consecutive floats per tile.
// Every mbarrier wait is bounded: a wait that gives up records
// SPC_ERR_TIMEOUT, the warp stops waiting (it keeps its loop so every
// barrier is still reached), and in-flight copies and MMAs are waited for
// (bounded) before the tensor memory is released.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "spc_device.cuh"
#include "spc_internal.h"
#include "spc_tc.cuh"

namespace spc {

constexpr int kTcRows = 128;                 // positions per tile
constexpr int kTcStages = 6;
constexpr uint32_t kTcTileBytes = kTcRows * kRowBytes;      // 32 KiB
constexpr uint32_t kTcHalfBytes = kTcTileBytes / 2;         // one 64-dim box
constexpr long long kTcWait = 4000000000ll;  // clock cycles (~2 s)

enum { kPassLse = 0, kPassScore = 1 };

template <int G, int PASS>
struct TcShape {
  // epilogue warps: CG column groups of 4 (one warp per TMEM lane quadrant each)
  static constexpr int CG = PASS == kPassLse ? G / 16 : (G >= 64 ? 2 : 1);
  static constexpr int kEpi = 128 * CG;
  static constexpr int kThreads = 64 + kEpi;
  // pass 1: D[128 query rows][128 positions], the 2G rows (head h high at 2h,
  // low at 2h + 1) repeated R times; each (replica, column group) takes CW
  // consecutive positions, split in two between the lanes of a high/low pair
  static constexpr int R = 64 / G;                                  // 1, 2, 4
  static constexpr int CW = kTcRows / (R * CG);                     // 32
  static constexpr int PPT = R * CG;                                // partials per (head, tile): 4
  // pass 2: D[128 positions][2G] (q high | q low); each thread one position, HPT heads
  static constexpr int HPT = G / CG;                                // 32 (G = 32, 64) or 16
  static constexpr int NCOL = PASS == kPassLse ? kTcRows : 2 * G;   // accumulator columns
  static constexpr int kQRows = PASS == kPassLse ? 128 : 2 * G;
  static constexpr uint32_t kQBytes = (uint32_t)kQRows * kRowBytes; // two swizzled 64-dim halves
  static constexpr uint32_t kXch = 2 * kTcRows * 4;                 // pass 2: column-group maxima, 2 buffers
  static constexpr int kTmemCols = 2 * NCOL < 32 ? 32 : 2 * NCOL;   // two accumulators
  static constexpr size_t kSmem = 1024 /* alignment slack */ + (size_t)kTcStages * kTcTileBytes + kQBytes +
                                  kXch + 16 * sizeof(uint64_t) + 16;
  // instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major
  static constexpr uint32_t kIdesc =
      PASS == kPassLse ? umma_idesc_bf16(128, kTcRows, false) : umma_idesc_bf16(kTcRows, 2 * G, false);
};

static_assert(TcShape<16, kPassLse>::PPT == 4 && TcShape<32, kPassLse>::PPT == 4 && TcShape<64, kPassLse>::PPT == 4,
              "one partial per (head, tile, quarter of the tile)");
int scan_tc_ppt(int G) {
  (void)G;
  return 4;
}

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
  asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
               :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
               : "memory");
}

template <int NT>
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, %0;" :: "n"(NT) : "memory"); }

__device__ __forceinline__ int tc_len(const int32_t* len, int b, int append, int cap) {
  int L = len[b];
  L = L < 0 ? 0 : (L > cap ? cap : L);
  return (append && L < cap) ? L + 1 : L;
}

// 2^x by the MUFU approximation (relative error ~2^-22, far inside the
// scores' tolerance); 2^-inf = 0
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// (max, sum of 2^(x - max)) merge with one exp2: the smaller maximum's sum is
// scaled; an empty side is (-inf, 0)
__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
  const bool keep = m >= m2;
  const float M = keep ? m : m2, mn = keep ? m2 : m;
  const float sb = keep ? s : s2, ss = keep ? s2 : s;
  s = mn == -INFINITY ? sb : sb + ss * ex2_approx(mn - M);
  m = M;
}

// ---------------------------------------------------------------- work split
// The tiles of one CTA. While every non-empty segment can have a CTA of its
// own, each segment gets 1 + (spare CTAs in proportion to its tile count)
// and its CTAs interleave: the c-th of n takes tiles c, c + n, c + 2n, ...
// (so that the CTAs of a segment read one advancing front of the cache, and
// no CTA changes queries mid-run). Otherwise the non-empty tiles of all
// segments, in order, are cut into equal consecutive runs. Every warp finds
// the CTA's start from the lengths, lane-parallel, and steps the same walk.
struct TileWalk {
  int seg, tile, step, count;   // step 0: consecutive run across segments
};

__device__ __forceinline__ int tc_seg_tiles(const ScanTcCall& a, int seg) {
  return (tc_len(a.len, seg / a.n_kv, a.append, a.cap) + kTcRows - 1) / kTcRows;
}

// Called by all 32 lanes of a warp: 32 segments at a time (prefix sums over
// the lanes), so a launch over hundreds of segments stays cheap.
__device__ TileWalk tile_walk(const ScanTcCall& a) {
  const int lane = threadIdx.x & 31;
  const int nseg = a.B * a.n_kv;
  int tot = 0, busy = 0;
  for (int s = lane; s < nseg; s += 32) {
    const int nt = tc_seg_tiles(a, s);
    tot += nt;
    busy += nt > 0;
  }
  const long long total = __reduce_add_sync(0xffffffffu, tot);
  busy = __reduce_add_sync(0xffffffffu, busy);
  TileWalk w{0, 0, 0, 0};
  const int c = (int)blockIdx.x;
  if (total == 0) return w;
  if (busy <= (int)gridDim.x) {
    const long long spare = (long long)gridDim.x - busy;
    int first = 0;                        // CTAs given to the segments before this group of 32
    for (int s0 = 0; s0 < nseg; s0 += 32) {
      const int s = s0 + lane;
      const int nt = s < nseg ? tc_seg_tiles(a, s) : 0;
      const int n = nt == 0 ? 0 : (int)min((long long)nt, 1 + spare * nt / total);
      const int incl = warp_incl_scan(n);
      const int lo = first + incl - n;
      const uint32_t hit = __ballot_sync(0xffffffffu, n > 0 && c >= lo && c < lo + n);
      if (hit) {
        const int src = __ffs(hit) - 1;
        const int k = c - __shfl_sync(0xffffffffu, lo, src);
        const int ns = __shfl_sync(0xffffffffu, n, src), nts = __shfl_sync(0xffffffffu, nt, src);
        w.seg = s0 + src;
        w.tile = k;
        w.step = ns;
        w.count = (nts - k + ns - 1) / ns;
        return w;
      }
      first += __shfl_sync(0xffffffffu, incl, 31);
    }
    return w;
  }
  const long long per = (total + gridDim.x - 1) / gridDim.x;
  const long long v = (long long)c * per;
  if (v >= total) return w;
  long long before = 0;                   // tiles of the segments before this group of 32
  for (int s0 = 0; s0 < nseg; s0 += 32) {
    const int s = s0 + lane;
    const int nt = s < nseg ? tc_seg_tiles(a, s) : 0;
    const int incl = warp_incl_scan(nt);
    const long long lo = before + incl - nt;
    const uint32_t hit = __ballot_sync(0xffffffffu, nt > 0 && v >= lo && v < lo + nt);
    if (hit) {
      const int src = __ffs(hit) - 1;
      w.seg = s0 + src;
      w.tile = (int)(v - __shfl_sync(0xffffffffu, lo, src));
      w.count = (int)min(per, total - v);
      return w;
    }
    before += __shfl_sync(0xffffffffu, incl, 31);
  }
  return w;
}

// the next tile of the walk (called only while tiles remain)
__device__ __forceinline__ void walk_next(const ScanTcCall& a, TileWalk& w) {
  if (w.step > 0) {
    w.tile += w.step;
    return;
  }
  ++w.tile;
  while (w.tile >= tc_seg_tiles(a, w.seg)) {
    ++w.seg;
    w.tile = 0;
  }
}

// ---------------------------------------------------------------- query operand
// The group's queries scaled by log2(e)/sqrt(d), split into a bf16 high part
// and a bf16 low part (q.K keeps ~16 significant bits of q), K-major with the
// 128-byte swizzle: element (row n, dim k) sits in half k / 64 at byte
// n * 128 + (((k % 64) / 8) ^ (n % 8)) * 16 + (k % 8) * 2. Pass 1 (A operand,
// 128 rows): head h high at row 2h + 2G r, low at row 2h + 1 + 2G r, for
// each replica r; pass 2 (B operand, 2G rows): high at row h, low at G + h.
// Thread `tid` of `nthr` converts the units of 8 dims u0 + i nthr, i < NB:
// load() issues all their loads, store() converts and stores them.
template <int G, int PASS, int NB>
struct QStage {
  static constexpr int kUnits = G * 16;   // 16 units of 8 dims per head
  float4 xs[2 * NB];

  __device__ __forceinline__ void load(const float* qg, int u0, int nthr) {
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      const int unit = u0 + i * nthr;
      if (unit < kUnits) {
        const float* src = qg + (size_t)(unit >> 4) * kD + (unit & 15) * 8;
        xs[2 * i] = *reinterpret_cast<const float4*>(src);
        xs[2 * i + 1] = *reinterpret_cast<const float4*>(src + 4);
      }
    }
  }

  __device__ __forceinline__ void store(uint32_t q0, float qscale, int u0, int nthr) const {
    using S = TcShape<G, PASS>;
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      const int unit = u0 + i * nthr;
      if (unit >= kUnits) break;
      const int h = unit >> 4, half = (unit >> 3) & 1, u = unit & 7;
      const float v[8] = {xs[2 * i].x, xs[2 * i].y, xs[2 * i].z, xs[2 * i].w,
                          xs[2 * i + 1].x, xs[2 * i + 1].y, xs[2 * i + 1].z, xs[2 * i + 1].w};
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float p0 = v[2 * e] * qscale, p1 = v[2 * e + 1] * qscale;
        const float h0 = bf16_round(p0), h1 = bf16_round(p1);
        hi[e] = pack_bf16(h0, h1);
        lo[e] = pack_bf16(p0 - h0, p1 - h1);
      }
      const uint32_t hb = q0 + (uint32_t)half * (S::kQRows * 128);
      constexpr int kCopies = PASS == kPassLse ? S::R : 1;
#pragma unroll
      for (int r = 0; r < kCopies; ++r) {
        const int nh = PASS == kPassLse ? 2 * G * r + 2 * h : h;
        const int nl = PASS == kPassLse ? nh + 1 : h + G;
        const uint32_t ah = hb + (uint32_t)nh * 128 + (uint32_t)((u ^ (nh & 7)) << 4);
        const uint32_t al = hb + (uint32_t)nl * 128 + (uint32_t)((u ^ (nl & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" :: "r"(ah), "r"(hi[0]), "r"(hi[1]), "r"(hi[2]),
                     "r"(hi[3]) : "memory");
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" :: "r"(al), "r"(lo[0]), "r"(lo[1]), "r"(lo[2]),
                     "r"(lo[3]) : "memory");
      }
    }
  }
};

// the whole operand by one warp, a batch of 8 units per lane in flight
template <int G, int PASS>
__device__ __forceinline__ void stage_q_warp(uint32_t q0, const float* qg, float qscale, int lane) {
  QStage<G, PASS, 8> qs;
  for (int u0 = lane; u0 < G * 16; u0 += 8 * 32) {
    qs.load(qg, u0, 32);
    qs.store(q0, qscale, u0, 32);
  }
  // generic-proxy writes made visible to the tensor core's async proxy
  fence_proxy_async_smem();
}

template <int G, int PASS>
__global__ void __launch_bounds__(TcShape<G, PASS>::kThreads, 1) scan_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                                                                                ScanTcCall a) {
  using S = TcShape<G, PASS>;
  extern __shared__ uint8_t tc_raw[];
  // 1024-byte aligned base (the 128-byte swizzle repeats every 8 rows of 128 B)
  const uint32_t raw_addr = smem_u32(tc_raw);
  uint8_t* base = tc_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* stages = base;
  uint8_t* qsm = stages + (size_t)kTcStages * kTcTileBytes;
  float* xch = reinterpret_cast<float*>(qsm + S::kQBytes);           // [2][128]
  uint64_t* full = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(xch) + S::kXch);
  uint64_t* empty = full + kTcStages;
  uint64_t* acc_full = empty + kTcStages;     // [2]
  uint64_t* acc_empty = acc_full + 2;         // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
  const uint32_t q0 = smem_u32(qsm);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&kmap)) : "memory");
  const TileWalk w0 = tile_walk(a);          // every warp, lane-parallel (no block barrier)
  // The first segment's queries: every thread issues its loads before any
  // key copy (behind the copies of all SMs they would wait for
  // microseconds), thread 0 then starts the first copies, and the
  // conversion overlaps their latency.
  constexpr int kPro = (G * 16 + S::kThreads - 1) / S::kThreads;
  QStage<G, PASS, kPro> qs;
  if (w0.count > 0) {
    const int b = w0.seg / a.n_kv, g = w0.seg - b * a.n_kv;
    qs.load(a.q + ((size_t)b * a.n_q + (size_t)g * G) * kD, threadIdx.x, S::kThreads);
  }
  // producer state (thread 0): tiles issued, and the walk at the last one
  int p_it = 0;
  bool p_dead = false;
  TileWalk pw = w0;
  auto issue = [&](int s) {
    mbar_arrive_expect_tx(&full[s], kTcTileBytes);
    const uint32_t dst = smem_u32(stages + (size_t)s * kTcTileBytes);
    tma_load_3d(dst, &kmap, 0, pw.tile * kTcRows, pw.seg, &full[s]);
    tma_load_3d(dst + kTcHalfBytes, &kmap, 64, pw.tile * kTcRows, pw.seg, &full[s]);
  };
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&full[s], 1);        // the producer's expect_tx arrival (+ the copies' bytes)
      mbar_init(&empty[s], 1);       // one tcgen05.commit
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);    // one tcgen05.commit
      mbar_init(&acc_empty[i], S::kEpi / 32);   // one arrival per epilogue warp
    }
    fence_mbar_init();
    // the initialised barriers made visible to the copies' async proxy
    // before this thread issues them (no block barrier in between)
    fence_proxy_async_smem();
    // the ring starts empty: the first copies need no wait
    for (; p_it < kTcStages && p_it < w0.count; ++p_it) {
      if (p_it) walk_next(a, pw);
      issue(p_it);
    }
  }
  if (w0.count > 0) {
    qs.store(q0, a.qscale, threadIdx.x, S::kThreads);
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc<S::kTmemCols>(tmem_slot);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ================= TMA producer (one lane)
    if (lane == 0) {
      for (; p_it < w0.count && !p_dead; ++p_it) {
        walk_next(a, pw);
        const int s = p_it % kTcStages;
        const uint32_t ph = (p_it / kTcStages) & 1;
        if (!mbar_wait_bounded(&empty[s], ph ^ 1, kTcWait)) {
          set_status(a.status, SPC_ERR_TIMEOUT);
          p_dead = true;
          break;
        }
        issue(s);
      }
      // the copies still in flight land before the CTA may exit
      for (int k = max(0, p_it - kTcStages); k < p_it; ++k)
        mbar_wait_bounded(&full[k % kTcStages], (k / kTcStages) & 1, kTcWait);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================= query operand of later segments, and MMA issue
    int it = 0, cur_seg = w0.seg, last_it = -1;
    bool dead = false;
    TileWalk w = w0;
    for (int i = 0; i < w.count; ++i) {
      if (i) walk_next(a, w);
      if (w.seg != cur_seg) {
        // the MMAs that read the previous segment's queries must be done
        if (last_it >= 0 && !dead) {
          bool ok = true;
          if (lane == 0) ok = mbar_wait_bounded(&acc_full[last_it & 1], (last_it >> 1) & 1, kTcWait);
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          if (!ok) {
            if (lane == 0) set_status(a.status, SPC_ERR_TIMEOUT);
            dead = true;
          }
        }
        const int b = w.seg / a.n_kv, g = w.seg - b * a.n_kv;
        stage_q_warp<G, PASS>(q0, a.q + ((size_t)b * a.n_q + (size_t)g * G) * kD, a.qscale, lane);
        __syncwarp();
        cur_seg = w.seg;
      }
      const int s = it % kTcStages;
      const uint32_t ph = (it / kTcStages) & 1;
      const int acc = it & 1;
      if (lane == 0 && !dead) {
        if (!mbar_wait_bounded(&full[s], ph, kTcWait) ||
            !mbar_wait_bounded(&acc_empty[acc], ((it >> 1) & 1) ^ 1, kTcWait)) {
          set_status(a.status, SPC_ERR_TIMEOUT);
          dead = true;
        } else {
          tc_fence_after();
          const uint32_t kst = smem_u32(stages + (size_t)s * kTcTileBytes);
          const uint32_t dcol = tmem + (uint32_t)(acc * S::NCOL);
          // K = 16 per instruction, 8 per tile; pass 1: D[q rows][positions] =
          // Q x K_tile^T, pass 2: D[positions][q rows] = K_tile x Q^T
#pragma unroll
          for (int half = 0; half < 2; ++half)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t kd = umma_desc_sw128(kst + (uint32_t)half * kTcHalfBytes + (uint32_t)k * 32);
              const uint64_t qd = umma_desc_sw128(q0 + (uint32_t)half * (S::kQRows * 128) + (uint32_t)k * 32);
              if constexpr (PASS == kPassLse)
                umma_f16(dcol, qd, kd, S::kIdesc, (half | k) ? 1u : 0u);
              else
                umma_f16(dcol, kd, qd, S::kIdesc, (half | k) ? 1u : 0u);
            }
          umma_commit(&empty[s]);          // the key stage may be refilled once these MMAs are done
          umma_commit(&acc_full[acc]);     // the accumulator is ready for the epilogue
          last_it = it;
        }
      }
      dead = __shfl_sync(0xffffffffu, dead ? 1 : 0, 0) != 0;
      last_it = __shfl_sync(0xffffffffu, last_it, 0);
      ++it;
    }
    // every MMA issued has completed before the tensor memory is released
    if (lane == 0 && last_it >= 0)
      mbar_wait_bounded(&acc_full[last_it & 1], (last_it >> 1) & 1, kTcWait);
    __syncwarp();
  } else {
    // ================= epilogue
    const int quad = warp & 3;                      // TMEM lanes 32 quad .. 32 quad + 31
    const int cg = (warp - 2) >> 2;                 // column group
    const uint32_t trow = tmem + ((uint32_t)(quad * 32) << 16);
    float lse_r[S::HPT];                            // pass 2: this thread's heads' normalisers
    int cur_seg = -1;
    bool dead = false;
    TileWalk w = w0;
    for (int it = 0; it < w.count; ++it) {
      if (it) walk_next(a, w);
      const int seg = w.seg, tile = w.tile;
      const int b = seg / a.n_kv, g = seg - b * a.n_kv;
      const int row0 = tile * kTcRows;
      const int nrows = min(kTcRows, tc_len(a.len, b, a.append, a.cap) - row0);
      if (PASS == kPassScore && seg != cur_seg) {
        const float* lg = a.lse + (size_t)b * a.n_q + (size_t)g * G + cg * S::HPT;
#pragma unroll
        for (int h = 0; h < S::HPT; ++h) lse_r[h] = lg[h];
        cur_seg = seg;
      }
      const int acc = it & 1;
      if (!dead && !mbar_wait_bounded(&acc_full[acc], (it >> 1) & 1, kTcWait)) {
        if (lane == 0) set_status(a.status, SPC_ERR_TIMEOUT);
        dead = true;
      }
      tc_fence_after();

      if constexpr (PASS == kPassLse) {
        // ---- lane = query row 32 quad + lane: head ((32 quad + lane) % 2G) / 2,
        // the high part on even lanes, the low part on odd ones; the warp's
        // CW = 32 columns are positions, the pair splits them: the even lane
        // takes the first 16 (its high part + its partner's low part), the
        // odd lane the last 16. Each thread folds its 16 into (max, sum
        // 2^(l - max)) with independent partial chains, and the pair merges.
        constexpr int CT = S::CW / 2;                 // positions per thread
        const int rep = quad * 16 / G;                // replica of this quadrant's rows
        const int slot = rep * S::CG + cg;            // quarter of the tile
        const int cbase = slot * S::CW;
        const bool odd = (lane & 1) != 0;
        float x[S::CW];
        if (!dead) {
          tmem_ld32(trow + (uint32_t)(acc * S::NCOL + cbase), x);
          tmem_ld_wait();
        }
        // this warp is done with the accumulator
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[acc]);
        float v[CT];
#pragma unroll
        for (int j = 0; j < CT; ++j) {
          const float send = odd ? x[j] : x[CT + j];
          const float mine = odd ? x[CT + j] : x[j];
          v[j] = mine + __shfl_xor_sync(0xffffffffu, send, 1);
        }
        const int nv = dead ? 0 : nrows - cbase - (odd ? CT : 0);   // valid positions of this thread's CT
        if (nv < CT) {
#pragma unroll
          for (int j = 0; j < CT; ++j) v[j] = j < nv ? v[j] : -INFINITY;
        }
        float m4[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) m4[k] = fmaxf(fmaxf(v[k], v[k + 4]), fmaxf(v[k + 8], v[k + 12]));
        float m = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        float sm = 0.f;
        if (m != -INFINITY) {
          float s4[4];
#pragma unroll
          for (int k = 0; k < 4; ++k)
            s4[k] = (ex2_approx(v[k] - m) + ex2_approx(v[k + 4] - m)) +
                    (ex2_approx(v[k + 8] - m) + ex2_approx(v[k + 12] - m));
          sm = (s4[0] + s4[1]) + (s4[2] + s4[3]);
        }
        lse_merge(m, sm, __shfl_xor_sync(0xffffffffu, m, 1), __shfl_xor_sync(0xffffffffu, sm, 1));
        if (!odd) {
          const int h = ((32 * quad + lane) % (2 * G)) >> 1;
          a.part[((size_t)b * a.n_q + (size_t)g * G + h) * a.n_parts + (size_t)tile * S::PPT + slot] =
              make_float2(m, sm);
        }
      } else {
        // ---- lane = position 32 quad + lane of the tile, HPT of the heads;
        // log2 of the group score: max over heads of l_h - lse_h
        const int p = quad * 32 + lane;
        const bool valid = p < nrows && !dead;
        float gs = -INFINITY;
        {
          const uint32_t hc = trow + (uint32_t)(acc * S::NCOL + cg * S::HPT);
          float hi[S::HPT], lo[S::HPT];
          if (!dead) {
            if constexpr (S::HPT == 32) {
              tmem_ld32(hc, hi);
              tmem_ld32(hc + G, lo);
            } else {
              tmem_ld16(hc, hi);
              tmem_ld16(hc + G, lo);
            }
            tmem_ld_wait();
          }
          // this warp is done with the accumulator
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[acc]);
#pragma unroll
          for (int h = 0; h < S::HPT; ++h) gs = fmaxf(gs, hi[h] + lo[h] - lse_r[h]);
        }
        if constexpr (S::CG == 2) {
          float* x = xch + (it & 1) * kTcRows;
          if (cg == 1) x[p] = gs;
          epi_bar<S::kEpi>();
          if (cg == 0) gs = fmaxf(gs, x[p]);
        }
        if (cg == 0 && valid) a.gscore[(size_t)seg * a.lstride + row0 + p] = gs;
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<S::kTmemCols>(tmem);
  }
}

// Normalisers from the pass-1 partials, one warp per (request, query head),
// eight partials in flight per lane: lse[b][h] = log2 sum_p 2^(l_h(p)) over
// p < len (INFINITY for an empty context). The first CTA of every (request,
// KV head) also writes the partials of a zero normaliser for the radix
// select that ranks the group scores (one partial per tile: (0, 1) first).
constexpr int kFoldThreads = 256;
constexpr int kFoldHeads = kFoldThreads / 32;     // heads per CTA
__global__ void __launch_bounds__(kFoldThreads) lse_fold_kernel(ScanTcCall a, int G, int ppt, float2* part1,
                                                                int n_parts1) {
  const int per_seg = (G + kFoldHeads - 1) / kFoldHeads;
  const int seg = blockIdx.x / per_seg, hblk = blockIdx.x - seg * per_seg;
  const int b = seg / a.n_kv, g = seg - b * a.n_kv;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int L = tc_len(a.len, b, a.append, a.cap);
  const int nv = ((L + kTcRows - 1) / kTcRows) * ppt;
  const int h = hblk * kFoldHeads + warp;
  if (h < G) {
    const float2* ph = a.part + ((size_t)b * a.n_q + (size_t)g * G + h) * a.n_parts;
    float m = -INFINITY, s = 0.f;
    for (int i0 = lane; i0 < nv; i0 += 32 * 8) {
      float2 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = i0 + 32 * u < nv ? __ldcg(ph + i0 + 32 * u) : make_float2(-INFINITY, 0.f);
#pragma unroll
      for (int u = 0; u < 8; ++u) lse_merge(m, s, v[u].x, v[u].y);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
      lse_merge(m, s, m2, s2);
    }
    if (lane == 0) a.lse[(size_t)b * a.n_q + (size_t)g * G + h] = s > 0.f ? m + log2f(s) : INFINITY;
  }
  if (hblk == 0)
    for (int t = threadIdx.x; t < n_parts1; t += kFoldThreads)
      part1[(size_t)seg * n_parts1 + t] = t == 0 ? make_float2(0.f, 1.f) : make_float2(-INFINITY, 0.f);
}

// ---------------------------------------------------------------- host side
template <int G, int PASS>
static cudaError_t launch_tc(const CUtensorMap& map, const ScanTcCall& c, int grid, cudaStream_t st) {
  const size_t smem = TcShape<G, PASS>::kSmem;
  cudaError_t e =
      set_func_attr((const void*)scan_tc_kernel<G, PASS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  scan_tc_kernel<G, PASS><<<grid, TcShape<G, PASS>::kThreads, smem, st>>>(map, c);
  return cudaGetLastError();
}

static int scan_tc_pass(ScanTcCall c, int G, int pass, cudaStream_t st) {
  // K_dlm as [segment = b * n_kv + g][position][dim], boxes of 128 positions x 64 dims
  CUtensorMap map;
  const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)c.cap, (uint64_t)c.B * c.n_kv};
  const uint64_t strides[2] = {(uint64_t)kRowBytes, (uint64_t)c.cap * kRowBytes};
  const uint32_t box[3] = {64, (uint32_t)kTcRows, 1};
  if (!tensor_map_bf16_sw128(&map, c.K, 3, dims, strides, box)) return SPC_ERR_CUDA;
  // one wave: one CTA per SM (at most one per capacity tile); each CTA
  // finds its tiles from the lengths on the device
  const int sms = device_sm_count() > 0 ? device_sm_count() : 1;
  const int grid = c.total_tiles < sms ? c.total_tiles : sms;
  if (grid < 1) return SPC_OK;
  cudaError_t e;
  switch (G * 2 + pass) {
    case 32 + kPassLse: e = launch_tc<16, kPassLse>(map, c, grid, st); break;
    case 32 + kPassScore: e = launch_tc<16, kPassScore>(map, c, grid, st); break;
    case 64 + kPassLse: e = launch_tc<32, kPassLse>(map, c, grid, st); break;
    case 64 + kPassScore: e = launch_tc<32, kPassScore>(map, c, grid, st); break;
    case 128 + kPassLse: e = launch_tc<64, kPassLse>(map, c, grid, st); break;
    case 128 + kPassScore: e = launch_tc<64, kPassScore>(map, c, grid, st); break;
    default: return SPC_ERR_SHAPE;
  }
  return e == cudaSuccess ? SPC_OK : SPC_ERR_CUDA;
}

int scan_tc_launch(ScanTcCall c, int G, void* stream) {
  return scan_tc_pass(c, G, kPassLse, static_cast<cudaStream_t>(stream));
}

int scan_tc_scores_launch(ScanTcCall c, int G, float2* part1, int n_parts1, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  lse_fold_kernel<<<c.B * c.n_kv * ((G + kFoldHeads - 1) / kFoldHeads), kFoldThreads, 0, st>>>(c, G, scan_tc_ppt(G), part1, n_parts1);
  if (cudaGetLastError() != cudaSuccess) return SPC_ERR_CUDA;
  return scan_tc_pass(c, G, kPassScore, st);
}

}  // namespace spc
