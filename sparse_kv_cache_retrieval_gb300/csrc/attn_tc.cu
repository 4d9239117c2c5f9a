// Sparse decode attention for groups of 64 query heads on one KV head (the
// MQA shape) on the 5th-generation tensor cores.
//
// Method: "ASPLOS'26 | SpeContext 让小模型先圈出重要 KV Cache" (marsggbo blog)
// §2 (softmax(q K^T / sqrt(d)) V over the kept Top-K rows only) and §4 (the
// LLM forward runs on the sparse KV prepared for this step); "SpeContext:
// Enabling Efficient Long-context Reasoning with Speculative Context Sparsity
// in LLMs" (paperlayer.ai summary) §4.3 (the selected KV serves every query
// head of its group).
//
// Per (layer, request, KV head) -- a segment -- the kept rows make a dense
// contraction: 64 query heads x 128 dims against up to 4096 K/V rows, twice
// (S = Q K^T, O = P V). It is HBM-bound (512 B of K and V per kept row);
// on the legacy mma.sync path its instruction stream held it near a fifth of
// the memory rate, so here both products run on tcgen05 with the
// accumulators in tensor memory.
//
// Tiles of 128 kept rows. For each tile:
//  * S[128][128] = Q2 K^T (M = 128, N = 128 rows, K = 128 dims): Q2 is the
//    group's 64 query rows written twice (rows h and h + 64 are both head h),
//    so that the same tile shape carries the two bf16 parts of P below. Q2
//    sits in tensor memory (the A operand of tcgen05.mma may live there), in
//    two buffers by segment parity, written by the softmax threads one
//    segment ahead.
//  * Softmax in base 2 by 8 warps: TMEM lane (row) r is read by two warps,
//    each taking 32 of the 64 kept rows [64 (r / 64), +64) of head r % 64, so
//    every logit is exponentiated once. The four threads of a head (in warps
//    q, q + 2, q + 4, q + 6) exchange their maxima through shared memory and
//    keep one running maximum, raised only when a tile's maximum exceeds it
//    by more than 8 (weights stay <= 2^8); then l and the head's accumulator
//    rows are rescaled.
//  * P (fp32) is split into two bf16 parts by bit selection -- the top 16
//    bits of p, then the top 16 bits of the (exact) remainder -- and written
//    to shared memory as the A operand: rows [0, 64) the high parts, rows
//    [64, 128) the low parts (K-major, 128-byte swizzle), so the weights keep
//    ~16 bits. One P buffer: the softmax of tile t + 1 writes it once the O
//    of tile t has read it (a second buffer, which lets the softmax run a
//    tile further ahead, measured 2-3% slower).
//  * O[128][128] += P V (M = 128, N = 128 dims, K = 128 rows; V is an
//    MN-major operand). Head h's output is O[h] + O[h + 64] divided by l.
// The products of bf16 operands are exact in the fp32 accumulators.
//
// K and V tiles come in by TMA, through tensor maps of the segment's view
// that each producer writes at the start of a segment (base address and row
// count patched into a host-made template with tensormap.replace, copied to a
// per-CTA global slot): a tiled copy of 128 contiguous rows when the view
// holds its kept rows in slots and every row of the tile is kept; otherwise
// row gathers (tile::gather4, four rows an instruction, from a map whose box
// is one row high) of the kept positions, a row not kept given a coordinate
// past the view's end so that the copy zero-fills it.
//
// Warp roles in one CTA per SM (persistent: a contiguous run of tiles, which
// may cover the end of one segment and the start of the next):
//  * warps 0-7: softmax, the Q2 operand and the segment epilogue (two warps
//    per TMEM lane quadrant);
//  * warps 8, 9: K and V producers, each a 2-slot ring of 32 KiB tiles;
//  * warp 10: allocates tensor memory (S in two buffers, O, Q2 in two), one
//    lane issues the MMAs in the order the softmax frees their inputs: O of
//    tile t as soon as its P is written, then S of tile t + 2 (S runs two
//    tiles ahead of the softmax).
// A segment split over several CTAs leaves one partial (m, l, O) per CTA in
// the workspace; the last CTA to finish merges them in CTA order
// (deterministic).
// Every wait is bounded: one that gives up records SPC_ERR_TIMEOUT, and the
// warp stops waiting but keeps its loop, so every barrier is still reached;
// copies in flight land and MMAs complete before the CTA releases its
// tensor memory.
#include <cuda.h>
#include <cuda_runtime.h>

#include "spc_device.cuh"
#include "spc_internal.h"
#include "spc_tc.cuh"

namespace spc {

constexpr int kAtG = 64;                              // query heads per KV head
constexpr int kAtRows = 128;                          // kept rows per tile
constexpr uint32_t kAtTile = kAtRows * kRowBytes;     // 32 KiB: a K, V, Q2 or P operand
constexpr uint32_t kAtBlock = kAtTile / 2;            // one 64-wide block of the 128-byte swizzle
constexpr int kAtKSlots = 2;                          // depth of the K ring
constexpr int kAtVSlots = 2;                          // depth of the V ring
constexpr int kAtPBufs = 1;                           // P operand buffers
constexpr int kAtSoftWarps = 8;
constexpr int kAtSoft = 32 * kAtSoftWarps;
constexpr int kAtKq = kAtSoftWarps / 4;              // warps per TMEM lane quadrant
constexpr int kAtKT = 64 / kAtKq;                     // kept rows of a tile per softmax thread
constexpr int kAtOT = kD / kAtKq;                     // O columns per softmax thread (epilogue, rescale)
constexpr int kAtWarpK = kAtSoftWarps, kAtWarpV = kAtSoftWarps + 1, kAtWarpMma = kAtSoftWarps + 2;
constexpr int kAtThreads = 32 * (kAtSoftWarps + 3);
constexpr float kAtHeadroom = 8.f;                    // log2 growth allowed before the maximum is raised
constexpr int kAtTmemCols = 512;                      // S0, S1, O, then Q2 in two 64-column buffers
constexpr uint32_t kAtColO = 256;
constexpr uint32_t kAtColQ = 384;
constexpr int kAtPart = kD + 4;                       // partial row: (m, l, pad, pad, O[128])
constexpr uint32_t kIdescS = umma_idesc_bf16(128, kAtRows, false);   // Q2 K^T: K-major
constexpr uint32_t kIdescO = umma_idesc_bf16(128, kD, true);         // P V: V is MN-major
constexpr uint32_t kAtMapBytes = 128;                 // one CUtensorMap

// shared memory, from a 1024-byte aligned base
constexpr uint32_t kAtOffK = 0;
constexpr uint32_t kAtOffV = kAtOffK + kAtKSlots * kAtTile;
constexpr uint32_t kAtOffP = kAtOffV + kAtVSlots * kAtTile;     // [kAtPBufs] P buffers
constexpr uint32_t kAtOffMap = kAtOffP + kAtPBufs * kAtTile;      // [2] tensor maps being patched
constexpr uint32_t kAtOffX = kAtOffMap + 2 * kAtMapBytes;         // [2 tiles][kAtKq][128] maxima
constexpr uint32_t kAtOffL = kAtOffX + 2 * kAtKq * kAtRows * 4;   // [2][kAtKq][64] partial sums of l
constexpr uint32_t kAtOffBar = kAtOffL + 2 * kAtKq * kAtG * 4;
constexpr int kAtBars = 2 * kAtKSlots + 2 * kAtVSlots + 2 + 2 + 2 + 2 * kAtPBufs + 1;   // see the list in the kernel
constexpr size_t kAtSmem = 1024 + kAtOffBar + kAtBars * 8 + 16;

int attn_tc_group() { return kAtG; }

// Tiling of one launch: nt tiles per segment, tpc tiles per CTA, at most
// max_pieces CTAs per segment. Runs of whole segments when they still keep
// 80% of the CTA target busy (no segment is then split, so no partials are
// merged); otherwise the tiles are spread evenly over the target. With one
// segment per CTA and CTAs to spare, split_pos lets the kernel give each
// segment whose view is read by position (row gathers, about twice a tiled
// copy's time per tile) two CTAs, one per half of its tiles. The CTA count is
// a fixed target (one per SM of a 152-SM GB300), not the device's, so the
// workspace size is a function of the shapes alone.
constexpr int kAtCtaTarget = 152;
static void attn_tc_plan(int n_layers, int B, int n_kv, int budget, int* nt, int* tpc, int* grid,
                         int* max_pieces, int* split_pos = nullptr) {
  const long long nseg = (long long)n_layers * B * n_kv;
  const int t = (budget + kAtRows - 1) / kAtRows;
  const long long total = nseg * t;
  const long long spc = (nseg + kAtCtaTarget - 1) / kAtCtaTarget;       // whole segments a CTA
  long long c;
  if ((nseg + spc - 1) / spc * 5 >= 4LL * kAtCtaTarget) {
    c = spc * t;
  } else {
    c = (total + kAtCtaTarget - 1) / kAtCtaTarget;
    if (c < 1) c = 1;
  }
  *nt = t;
  *tpc = (int)c;
  *grid = (int)((total + c - 1) / c);
  const int mp = c % t == 0 ? 1 : (t + (int)c - 1) / (int)c + 1;
  *max_pieces = mp < t ? mp : t;
  const bool sp = c == t && nseg < kAtCtaTarget && t >= 2;
  if (split_pos) *split_pos = sp ? 1 : 0;
  if (sp) {
    *grid = (int)(2 * nseg < kAtCtaTarget ? 2 * nseg : kAtCtaTarget);
    *max_pieces = 2;
  }
}

__device__ __forceinline__ void soft_bar() { asm volatile("bar.sync 1, %0;" :: "n"(kAtSoft) : "memory"); }
// the softmax warps that hold the same heads (lane quadrants q and q + 2 for
// q = warp % 2): named barrier 2 + warp % 2
__device__ __forceinline__ void head_bar(int warp) {
  if (warp & 1)
    asm volatile("bar.sync 3, %0;" :: "n"(kAtSoft / 2) : "memory");
  else
    asm volatile("bar.sync 2, %0;" :: "n"(kAtSoft / 2) : "memory");
}

// A bounded wait by every lane of a warp with one warp-wide verdict, so that
// the warp-collective tcgen05.ld / tcgen05.st that follow stay convergent.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, long long limit) {
  return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, limit));
}

// 2^x for x <= 8 (and -inf -> 0): the MUFU approximation, relative error
// ~2^-22, far inside what the bf16 split of the weights keeps
__device__ __forceinline__ float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Both index entries of kept index i (selected position, slot map entry),
// fetched one tile ahead; i >= K reads nothing
struct AtIdx {
  int sel, slot;
};
__device__ __forceinline__ AtIdx at_fetch(const int32_t* sel, const int32_t* slot, int i, int K) {
  AtIdx x{-1, -1};
  if (i < K) {
    x.sel = __ldg(sel + i);
    x.slot = __ldg(slot + i);
  }
  return x;
}
// Row of kept index i: the slot i (slot views) or the position selected[i]
// (full-cache views); -1 when the index keeps nothing.
__device__ __forceinline__ int at_row(bool use_slots, long long rows, AtIdx x, int i) {
  const int v = use_slots ? x.slot : x.sel;
  if (v < 0) return -1;
  const long long r = use_slots ? (long long)i : (long long)v;
  return r < rows ? (int)r : -1;
}

// Segment and tile of global tile t; at_next steps to t + 1 without divisions
struct AtTile {
  int seg, tile, lb, g, b;
};
__device__ __forceinline__ AtTile at_tile(const AttnTcCall& a, int t) {
  AtTile x;
  x.seg = t / a.nt;
  x.tile = t - x.seg * a.nt;
  x.lb = x.seg / a.n_kv;
  x.g = x.seg - x.lb * a.n_kv;
  x.b = x.lb % a.B;
  return x;
}
__device__ __forceinline__ void at_next(const AttnTcCall& a, AtTile& x) {
  if (++x.tile < a.nt) return;
  x.tile = 0;
  ++x.seg;
  if (++x.g < a.n_kv) return;
  x.g = 0;
  ++x.lb;
  if (++x.b == a.B) x.b = 0;
}

// Q2 of segment `seg` for this thread's TMEM lane (head h) and dims
// [kAtOT cq, +kAtOT): bf16 pairs, loaded first, stored to tensor memory once
// the buffer is free
struct AtQ {
  uint32_t w[kAtOT / 2];
};
__device__ __forceinline__ void at_q_load(const AttnTcCall& a, int seg, int h, int cq, AtQ& q) {
  const int lb = seg / a.n_kv, g = seg - lb * a.n_kv;
  const uint4* src = reinterpret_cast<const uint4*>(a.q + ((size_t)lb * a.n_q + (size_t)g * kAtG + h) * kD + kAtOT * cq);
#pragma unroll
  for (int i = 0; i < kAtOT / 8; ++i) {
    const uint4 v = ldg_stream(src + i);
    q.w[4 * i] = v.x; q.w[4 * i + 1] = v.y; q.w[4 * i + 2] = v.z; q.w[4 * i + 3] = v.w;
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* map, int x, int y, uint64_t* bar) {
  asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
               :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)) : "memory");
}
// rows y0..y3 (64 elements from column x of each) to four consecutive
// 128-byte rows at dst; the map's box is one row high
__device__ __forceinline__ void tma_gather4(uint32_t dst, const void* map, int x, int y0, int y1, int y2, int y3,
                                            uint64_t* bar) {
  asm volatile("cp.async.bulk.tensor.2d.shared::cta.global.tile::gather4.mbarrier::complete_tx::bytes"
               " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];"
               :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3),
                  "r"(smem_u32(bar)) : "memory");
}

// Registers per thread capped so that the CTA leaves room on the SM for a CTA
// of the gather kernel (128 threads x 128 registers), which runs beside this
// kernel in the decode step.
constexpr int kAtMaxReg = ((65536 - 128 * 128) / kAtThreads) & ~7;
__global__ void __maxnreg__(kAtMaxReg) attn_tc_kernel(const __grid_constant__ CUtensorMap tile_tmpl,
                                                const __grid_constant__ CUtensorMap row_tmpl,
                                                AttnTcCall a) {
  extern __shared__ uint8_t at_raw[];
  const uint32_t raw_addr = smem_u32(at_raw);
  uint8_t* base = at_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* kring = base + kAtOffK;
  uint8_t* vring = base + kAtOffV;
  uint8_t* pop = base + kAtOffP;
  uint8_t* smaps = base + kAtOffMap;
  float* xmax = reinterpret_cast<float*>(base + kAtOffX);
  float* xl = reinterpret_cast<float*>(base + kAtOffL);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + kAtOffBar);
  uint64_t* kfull = bars;                    // [kAtKSlots] TMA bytes
  uint64_t* kfree = kfull + kAtKSlots;       // [kAtKSlots] commit after the tile's S MMAs
  uint64_t* vfull = kfree + kAtKSlots;       // [kAtVSlots] TMA bytes
  uint64_t* vfree = vfull + kAtVSlots;       // [kAtVSlots] commit after the tile's O MMAs
  uint64_t* qfull = vfree + kAtVSlots;       // [2] 8 softmax-warp arrivals: Q2 of a segment written
  uint64_t* sfull = qfull + 2;               // [2] commit: S of the tile is in tensor memory
  uint64_t* sfree = sfull + 2;               // [2] 8 softmax-warp arrivals: S read
  uint64_t* pfull = sfree + 2;               // [kAtPBufs] 8 arrivals: P written (and O rescaled)
  uint64_t* pfree = pfull + kAtPBufs;        // [kAtPBufs] commit after the tile's O MMAs
  uint64_t* ofull = pfree + kAtPBufs;        // commit after a segment's last O MMAs
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ofull + 1);
  int* s_last = reinterpret_cast<int*>(tmem_slot + 1);
  __shared__ int s_run[4];                   // split_pos: this CTA's tiles and piece

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kAtKSlots; ++s) {
      mbar_init(&kfull[s], 1);
      mbar_init(&kfree[s], 1);
    }
    for (int s = 0; s < kAtVSlots; ++s) {
      mbar_init(&vfull[s], 1);
      mbar_init(&vfree[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&qfull[s], kAtSoftWarps);
      mbar_init(&sfull[s], 1);
      mbar_init(&sfree[s], kAtSoftWarps);
    }
    for (int s = 0; s < kAtPBufs; ++s) {
      mbar_init(&pfull[s], kAtSoftWarps);
      mbar_init(&pfree[s], 1);
    }
    mbar_init(ofull, 1);
    fence_mbar_init();
  }
  if (warp == kAtWarpMma) tmem_alloc<kAtTmemCols>(tmem_slot);
  if (a.split_pos && warp == 0) {
    // one segment per CTA, two for a segment whose view reads positions when
    // the grid has a CTA for every such segment (else none is split): this
    // CTA's (first tile, end, pieces, piece) from a prefix over the segments
    const int nseg = a.total / a.nt;
    auto by_pos = [&](int sg) { return sg < nseg && a.views[sg / a.n_kv].use_slots == 0; };
    int npos = 0;
    for (int s0 = 0; s0 < nseg; s0 += 32) npos += __popc(__ballot_sync(0xffffffffu, by_pos(s0 + lane)));
    const bool split = nseg + npos <= (int)gridDim.x;
    if (lane == 0) { s_run[0] = 0; s_run[1] = 0; s_run[2] = 1; s_run[3] = 0; }
    __syncwarp();
    const int cta = blockIdx.x, half = (a.nt + 1) / 2;
    int off = 0;
    for (int s0 = 0; s0 < nseg; s0 += 32) {
      const int sg = s0 + lane;
      const int n = sg < nseg ? 1 + ((split && by_pos(sg)) ? 1 : 0) : 0;
      const int incl = warp_incl_scan(n), first = off + incl - n;
      if (n > 0 && cta >= first && cta < first + n) {
        const int pc = cta - first;
        s_run[0] = sg * a.nt + (pc == 1 ? half : 0);
        s_run[1] = sg * a.nt + (n == 1 || pc == 1 ? a.nt : half);
        s_run[2] = n;
        s_run[3] = pc;
      }
      off += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  int t0 = blockIdx.x * a.tpc, t1 = min(a.total, t0 + a.tpc);
  int split_pieces = 1, split_piece = 0;
  if (a.split_pos) {
    t0 = s_run[0];
    t1 = s_run[1];
    split_pieces = s_run[2];
    split_piece = s_run[3];
  }

  if (warp == kAtWarpK || warp == kAtWarpV) {
    // ================= producers (K; V)
    const int op = warp - kAtWarpK;              // 0: K, 1: V
    const int nslots = op == 0 ? kAtKSlots : kAtVSlots;
    uint8_t* ring = op == 0 ? kring : vring;
    uint64_t* full = op == 0 ? kfull : vfull;
    uint64_t* empty = op == 0 ? kfree : vfree;
    uint8_t* smap = smaps + op * kAtMapBytes;
    // this CTA's global tensor-map slots: [operand][segment parity][tiled, row gather]
    uint8_t* gmaps = a.maps + ((size_t)blockIdx.x * 2 + op) * 4 * kAtMapBytes;
    bool dead = false;
#ifdef SPC_TEST_HOOKS
    // a starved launch: no copy is issued, so every consumer's wait runs out
    const bool starve = a.starve != 0;
#else
    constexpr bool starve = false;
#endif
    int cur_seg = -1, ns = -1, n_issued = 0;
    int map_seg_tile = -1, map_seg_row = -1;      // segment whose map each global slot holds
    spc_kv_view vw{};
    const uint16_t* src = nullptr;
    // row indices of the next tile, fetched one tile ahead
    AtIdx nx[4];
    AtTile y = at_tile(a, t0);
    if (t0 < t1) {
      const size_t ioff = ((size_t)y.b * a.n_kv + y.g) * a.K;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        nx[k] = at_fetch(a.selected + ioff, a.slot_pos + ioff, y.tile * kAtRows + 32 * k + lane, a.K);
    }
    for (int t = t0, it = 0; t < t1 && !starve; ++t, ++it) {
      const AtTile x = y;
      at_next(a, y);
      AtIdx cur[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) cur[k] = nx[k];
      if (t + 1 < t1) {
        const size_t ioff = ((size_t)y.b * a.n_kv + y.g) * a.K;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          nx[k] = at_fetch(a.selected + ioff, a.slot_pos + ioff, y.tile * kAtRows + 32 * k + lane, a.K);
      }
      if (x.seg != cur_seg) {
        cur_seg = x.seg;
        ++ns;
        vw = a.views[x.lb];
        src = static_cast<const uint16_t*>(op == 0 ? vw.k : vw.v) + (size_t)x.g * vw.rows * kD;
      }
      int row[4];
      bool all = true;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        row[k] = at_row(vw.use_slots != 0, vw.rows, cur[k], x.tile * kAtRows + 32 * k + lane);
        all = all && __all_sync(0xffffffffu, row[k] >= 0);
      }
      const int s = it % nslots;
      if (!dead && !mbar_wait_bounded(&empty[s], ((it / nslots) & 1) ^ 1, a.wait_limit)) {
        if (lane == 0) set_status(a.status, SPC_ERR_TIMEOUT);
        dead = true;
      }
      dead = __any_sync(0xffffffffu, dead);
      if (dead) continue;
      const uint32_t dst = smem_u32(ring + (size_t)s * kAtTile);
      const int kind = (vw.use_slots && all) ? 0 : 1;      // tiled copy, or row gathers
      const uint8_t* gmap = gmaps + (size_t)((ns & 1) * 2 + kind) * kAtMapBytes;
      if ((kind == 0 ? map_seg_tile : map_seg_row) != x.seg) {
        // this segment's map of this kind: the template with the view's base
        // address and row count, copied to the global slot of this parity.
        // The TMAs that used that slot (two segments ago) have landed: their
        // ring slots were released before the wait above returned.
        if (kind == 0) map_seg_tile = x.seg; else map_seg_row = x.seg;
        const CUtensorMap* tmpl = kind == 0 ? &tile_tmpl : &row_tmpl;
        if (lane < 8) reinterpret_cast<uint4*>(smap)[lane] = reinterpret_cast<const uint4*>(tmpl)[lane];
        __syncwarp();
        if (lane == 0) {
          asm volatile("tensormap.replace.tile.global_address.shared::cta.b1024.b64 [%0], %1;"
                       :: "r"(smem_u32(smap)), "l"(reinterpret_cast<uint64_t>(src)) : "memory");
          asm volatile("tensormap.replace.tile.global_dim.shared::cta.b1024.b32 [%0], 1, %1;"
                       :: "r"(smem_u32(smap)), "r"((uint32_t)vw.rows) : "memory");
        }
        __syncwarp();
        asm volatile(
            "tensormap.cp_fenceproxy.global.shared::cta.tensormap::generic.release.gpu.sync.aligned [%0], [%1], 128;"
            :: "l"(reinterpret_cast<uint64_t>(gmap)), "r"(smem_u32(smap)) : "memory");
        asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;"
                     :: "l"(reinterpret_cast<uint64_t>(gmap)) : "memory");
      }
      if (lane == 0) mbar_arrive_expect_tx(&full[s], kAtTile);
      if (kind == 0) {
        if (lane == 0) {
          tma_load_2d(dst, gmap, 0, x.tile * kAtRows, &full[s]);
          tma_load_2d(dst + kAtBlock, gmap, 64, x.tile * kAtRows, &full[s]);
        }
      } else {
        // lane L gathers the tile's rows 4L .. 4L + 3 into both 64-dim blocks;
        // a row not kept reads past the view's end (zero-filled)
        __syncwarp();
        int y[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int srcl = (4 * lane + i) & 31;
          const int v0 = __shfl_sync(0xffffffffu, row[0], srcl), v1 = __shfl_sync(0xffffffffu, row[1], srcl);
          const int v2 = __shfl_sync(0xffffffffu, row[2], srcl), v3 = __shfl_sync(0xffffffffu, row[3], srcl);
          const int k = lane >> 3;                 // (4 lane + i) / 32
          const int v = k == 0 ? v0 : k == 1 ? v1 : k == 2 ? v2 : v3;
          y[i] = v >= 0 ? v : (int)vw.rows;
        }
        const uint32_t d = dst + (uint32_t)(4 * lane) * 128;
        tma_gather4(d, gmap, 0, y[0], y[1], y[2], y[3], &full[s]);
        tma_gather4(d + kAtBlock, gmap, 64, y[0], y[1], y[2], y[3], &full[s]);
      }
      n_issued = it + 1;
    }
    // the copies still in flight land before the CTA may exit (they have,
    // unless a consumer gave up waiting)
    if (lane == 0) {
      for (int k = max(0, n_issued - nslots); k < n_issued; ++k)
        mbar_wait_bounded(&full[k % nslots], (k / nslots) & 1, a.wait_limit);
    }
    __syncwarp();
  } else if (warp == kAtWarpMma) {
    // ================= MMA issue (one lane)
    if (lane == 0) {
      bool dead = false;
      const uint32_t pa = smem_u32(pop);
      const uint32_t ka = smem_u32(kring), va = smem_u32(vring);
      // O for tile pt: P from the softmax, V from the ring
      auto issue_o = [&](int pt, bool first, bool last) {
        const int s = pt % kAtVSlots, pb = pt % kAtPBufs;
        if (!dead && (!mbar_wait_bounded(&pfull[pb], (pt / kAtPBufs) & 1, a.wait_limit) ||
                      !mbar_wait_bounded(&vfull[s], (pt / kAtVSlots) & 1, a.wait_limit))) {
          set_status(a.status, SPC_ERR_TIMEOUT);
          dead = true;
        }
        if (dead) return;
        tc_fence_after();
        const uint32_t vt = va + (uint32_t)s * kAtTile;
        const uint32_t pt_a = pa + (uint32_t)pb * kAtTile;
#pragma unroll
        for (int j = 0; j < kAtRows / 16; ++j) {
          const uint64_t ad = umma_desc_sw128(pt_a + (uint32_t)(j >> 2) * kAtBlock + (uint32_t)(j & 3) * 32);
          const uint64_t bd = umma_desc_sw128_mn(vt + (uint32_t)j * 16 * 128, kAtBlock);
          umma_f16(tmem + kAtColO, ad, bd, kIdescO, (first && j == 0) ? 0u : 1u);
        }
        umma_commit(&vfree[s]);
        umma_commit(&pfree[pb]);
        if (last) umma_commit(ofull);
      };
      // S for tile u (segment counter ns_u, first tile of its segment or not)
      auto issue_s = [&](int u, int ns_u, bool first) {
        if (first && !dead && !mbar_wait_bounded(&qfull[ns_u & 1], (ns_u >> 1) & 1, a.wait_limit)) {
          set_status(a.status, SPC_ERR_TIMEOUT);
          dead = true;
        }
        const int s = u % kAtKSlots, sb = u & 1;
        if (!dead && (!mbar_wait_bounded(&kfull[s], (u / kAtKSlots) & 1, a.wait_limit) ||
                      !mbar_wait_bounded(&sfree[sb], ((u >> 1) & 1) ^ 1, a.wait_limit))) {
          set_status(a.status, SPC_ERR_TIMEOUT);
          dead = true;
        }
        if (dead) return;
        tc_fence_after();
        const uint32_t kt = ka + (uint32_t)s * kAtTile;
        const uint32_t qa = tmem + kAtColQ + (uint32_t)(ns_u & 1) * (kD / 2);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint64_t bd = umma_desc_sw128(kt + (uint32_t)(kk >> 2) * kAtBlock + (uint32_t)(kk & 3) * 32);
          umma_f16_tmem_a(tmem + (uint32_t)sb * kAtRows, qa + (uint32_t)kk * 8, bd, kIdescS, kk ? 1u : 0u);
        }
        umma_commit(&kfree[s]);
        umma_commit(&sfull[sb]);
      };
      const int n = t1 - t0;
      const int tile0 = n > 0 ? t0 % a.nt : 0;     // tile of t0 within its segment
      // tile u of this CTA: first / last tile of a segment, segment counter
      auto is_first = [&](int u) { return u == 0 || (tile0 + u) % a.nt == 0; };
      auto is_last = [&](int u) { return u + 1 == n || (tile0 + u + 1) % a.nt == 0; };
      int ns_s = -1;                               // segment counter of the last S issued
      for (int u = 0; u < n && u < 2; ++u) {
        if (is_first(u)) ++ns_s;
        issue_s(u, ns_s, is_first(u));
      }
      for (int u = 0; u < n; ++u) {
        issue_o(u, is_first(u), is_last(u));
        if (u + 2 < n) {
          if (is_first(u + 2)) ++ns_s;
          issue_s(u + 2, ns_s, is_first(u + 2));
        }
      }
      // every MMA has completed before the tensor memory is released
      if (n > 0 && !dead) mbar_wait_bounded(&pfree[(n - 1) % kAtPBufs], ((n - 1) / kAtPBufs) & 1, a.wait_limit);
    }
    __syncwarp();
  } else {
    // ================= softmax and epilogue
    // warp w reads TMEM lanes 32 (w % 4) .. +31 (lane r: head r % 64) and
    // takes kAtKT kept rows of the tile: [64 (r / 64) + kAtKT (w / 4), +kAtKT)
    const int qd = warp & 3, cq = warp >> 2;
    const int r = qd * 32 + lane, h = r & (kAtG - 1), hf = r >> 6;
    const int col = 64 * hf + kAtKT * cq;              // this thread's first kept row in a tile
    const int kl = lane & (kAtKT - 1);                 // the kept row whose index this lane fetches
    const uint32_t trow = tmem + ((uint32_t)(qd * 32) << 16);
    bool dead = false;
    float m = -INFINITY, l = 0.f;
    int cur_seg = -1, ns = -1;
    spc_kv_view vw{};
    AtIdx nx{-1, -1};
    AtTile y = at_tile(a, t0);
    if (t0 < t1) {
      const size_t ioff = ((size_t)y.b * a.n_kv + y.g) * a.K;
      nx = at_fetch(a.selected + ioff, a.slot_pos + ioff, y.tile * kAtRows + col + kl, a.K);
      // Q2 of the first segment, buffer 0
      AtQ q;
      at_q_load(a, y.seg, h, cq, q);
      tmem_st_n<kAtOT / 2>(trow + kAtColQ + (uint32_t)(kAtOT / 2 * cq), q.w);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&qfull[0]);
    }
    for (int t = t0, it = 0; t < t1; ++t, ++it) {
      const AtTile x = y;
      at_next(a, y);
      const bool last = t + 1 == t1 || y.tile == 0;
      const AtIdx cur = nx;
      if (t + 1 < t1) {
        const size_t ioff = ((size_t)y.b * a.n_kv + y.g) * a.K;
        nx = at_fetch(a.selected + ioff, a.slot_pos + ioff, y.tile * kAtRows + col + kl, a.K);
      }
      // a new segment: Q2 of the next one (if this CTA has it) goes into the
      // other buffer once this tile's S is in (then every S of the segment
      // before, the buffer's last reader, has completed)
      const bool seg_start = x.seg != cur_seg;
      const bool q_next = seg_start && t + (a.nt - x.tile) < t1;
      if (seg_start) {
        cur_seg = x.seg;
        ++ns;
        vw = a.views[x.lb];
        m = -INFINITY;
        l = 0.f;
      }
      const uint32_t okm =
          __ballot_sync(0xffffffffu, at_row(vw.use_slots != 0, vw.rows, cur, x.tile * kAtRows + col + kl) >= 0);

      const int sb = it & 1;
      if (!dead && !warp_wait(&sfull[sb], (it >> 1) & 1, a.wait_limit)) {
        if (lane == 0) set_status(a.status, SPC_ERR_TIMEOUT);
        dead = true;
      }
      tc_fence_after();
      if (q_next) {
        if (!dead) {
          AtQ qn;
          at_q_load(a, x.seg + 1, h, cq, qn);
          tmem_st_n<kAtOT / 2>(trow + kAtColQ + (uint32_t)(((ns + 1) & 1) * (kD / 2) + kAtOT / 2 * cq), qn.w);
          tmem_st_wait();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&qfull[(ns + 1) & 1]);
      }
      float s[kAtKT];
      if (!dead) {
        tmem_ld_n<kAtKT>(trow + (uint32_t)sb * kAtRows + (uint32_t)col, s);
        tmem_ld_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sfree[sb]);
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      if (dead || okm != 0xffffffffu) {
#pragma unroll
        for (int j = 0; j < kAtKT; ++j) s[j] = (!dead && ((okm >> j) & 1u)) ? s[j] : -INFINITY;
      }
#pragma unroll
      for (int j = 0; j < kAtKT; ++j) mx4[j & 3] = fmaxf(mx4[j & 3], s[j]);
      const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      // the head's tile maximum (scaled to base 2) over its 2 kAtKq threads
      float* xm = xmax + sb * kAtKq * kAtRows;
      xm[cq * kAtRows + r] = mx * a.scale2;
      head_bar(warp);
      float M = -INFINITY;
#pragma unroll
      for (int c = 0; c < kAtKq; ++c) M = fmaxf(M, fmaxf(xm[c * kAtRows + r], xm[c * kAtRows + (r ^ 64)]));
      bool rescale = false;
      float alpha = 1.f;
      if (M > m + kAtHeadroom) {          // false for M = -inf; true for the first finite maximum
        if (m != -INFINITY) {
          alpha = ex2_fast(m - M);
          l *= alpha;
          rescale = true;                 // O already holds this segment's earlier tiles
        }
        m = M;
      }
      // P = 2^(s scale2 - m), in place
      float lsum = 0.f;
      if (m != -INFINITY) {
        float ls4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < kAtKT; ++j) {
          s[j] = ex2_fast(fmaf(s[j], a.scale2, -m));
          ls4[j & 3] += s[j];
        }
        lsum = (ls4[0] + ls4[1]) + (ls4[2] + ls4[3]);
      } else {
#pragma unroll
        for (int j = 0; j < kAtKT; ++j) s[j] = 0.f;
      }
      l += lsum;
      // the O MMAs of tile it - kAtPBufs are done: its P buffer may be overwritten
      if (!dead && !warp_wait(&pfree[it % kAtPBufs], ((it / kAtPBufs) & 1) ^ 1, a.wait_limit)) {
        if (lane == 0) set_status(a.status, SPC_ERR_TIMEOUT);
        dead = true;
      }
      const bool any_rescale = __any_sync(0xffffffffu, rescale);
      // O holds earlier tiles to rescale: the O MMAs of tile it - 1 must be done
      if (any_rescale && it > 0 && !dead &&
          !warp_wait(&pfree[(it - 1) % kAtPBufs], ((it - 1) / kAtPBufs) & 1, a.wait_limit)) {
        if (lane == 0) set_status(a.status, SPC_ERR_TIMEOUT);
        dead = true;
      }
      tc_fence_after();
      if (any_rescale && !dead) {
        // warp-wide (the accesses are collective); other heads scale by 1.
        // The warps of a lane quadrant take O's columns [kAtOT cq, +kAtOT).
#pragma unroll 1
        for (int c = 0; c < kAtOT / 32; ++c) {
          float o[32];
          const uint32_t oc = trow + kAtColO + (uint32_t)(kAtOT * cq + 32 * c);
          tmem_ld32(oc, o);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] *= alpha;
          tmem_st32(oc, o);
        }
        tmem_st_wait();
      }
      {
        // high parts (the top 16 bits of p) to row h, the top 16 bits of the
        // remainder to row h + 64, in the block of this thread's kept rows:
        // 16-byte unit u holds kept rows 8u .. 8u + 7
        const uint32_t pb = smem_u32(pop) + (uint32_t)(it % kAtPBufs) * kAtTile + (uint32_t)hf * kAtBlock;
#pragma unroll
        for (int uu = 0; uu < kAtKT / 8; ++uu) {
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t b0 = __float_as_uint(s[8 * uu + 2 * e]), b1 = __float_as_uint(s[8 * uu + 2 * e + 1]);
            hi[e] = __byte_perm(b0, b1, 0x7632);
            lo[e] = __byte_perm(__float_as_uint(s[8 * uu + 2 * e] - __uint_as_float(b0 & 0xffff0000u)),
                                __float_as_uint(s[8 * uu + 2 * e + 1] - __uint_as_float(b1 & 0xffff0000u)), 0x7632);
          }
          const int u = kAtKT / 8 * cq + uu;
          const uint32_t off = (uint32_t)(h * 128 + ((u ^ (h & 7)) << 4));
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" :: "r"(pb + off), "r"(hi[0]), "r"(hi[1]), "r"(hi[2]),
                       "r"(hi[3]) : "memory");
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" :: "r"(pb + off + kAtG * 128), "r"(lo[0]), "r"(lo[1]),
                       "r"(lo[2]), "r"(lo[3]) : "memory");
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&pfull[it % kAtPBufs]);

      if (!last) continue;
      // ---- segment epilogue: O_h = O[h] + O[h + 64], l_h = its four threads' sums
      if (!dead && !warp_wait(ofull, ns & 1, a.wait_limit)) {
        if (lane == 0) set_status(a.status, SPC_ERR_TIMEOUT);
        dead = true;
      }
      tc_fence_after();
      // the P buffer is free (every O MMA of the segment is done) until the
      // softmax threads write the next tile's P, which they do only after the
      // barrier that closes this epilogue: it holds the low rows
      float* xo = reinterpret_cast<float*>(pop);     // [64][128], float4 j of row h at (j + h) % 32
      xl[(hf * kAtKq + cq) * kAtG + h] = l;
      if (hf == 1) {
#pragma unroll 1
        for (int c = 0; c < kAtOT / 32; ++c) {
          float o[32];
          if (!dead) {
            tmem_ld32(trow + kAtColO + (uint32_t)(kAtOT * cq + 32 * c), o);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = 0.f;
          }
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4)
            reinterpret_cast<float4*>(xo + h * kD)[(kAtOT / 4 * cq + 8 * c + q4 + h) & 31] =
                make_float4(o[4 * q4], o[4 * q4 + 1], o[4 * q4 + 2], o[4 * q4 + 3]);
        }
      }
      tc_fence_before();
      soft_bar();
      const int pieces =
          a.split_pos ? split_pieces : (x.seg * a.nt + a.nt - 1) / a.tpc - (x.seg * a.nt) / a.tpc + 1;
      const int piece = a.split_pos ? split_piece : blockIdx.x - (x.seg * a.nt) / a.tpc;
      float* outp = a.out + ((size_t)x.lb * a.n_q + (size_t)x.g * kAtG + h) * kD;
      float* res = a.part + ((size_t)x.seg * a.max_pieces + piece) * (size_t)kAtG * kAtPart + (size_t)h * kAtPart;
      if (hf == 0) {
        tc_fence_after();
        float L = 0.f;
#pragma unroll
        for (int c = 0; c < 2 * kAtKq; ++c) L += xl[c * kAtG + h];
        const float li = L > 0.f ? 1.f / L : 0.f;
        if (pieces > 1 && cq == 0) {
          res[0] = m;
          res[1] = L;
        }
#pragma unroll 1
        for (int c = 0; c < kAtOT / 32; ++c) {
          float o[32];
          if (!dead) {
            tmem_ld32(trow + kAtColO + (uint32_t)(kAtOT * cq + 32 * c), o);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = 0.f;
          }
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {
            const int j4 = kAtOT / 4 * cq + 8 * c + q4;   // float4 index within the 128 dims
            const float4 lo4 = reinterpret_cast<const float4*>(xo + h * kD)[(j4 + h) & 31];
            float4 v = make_float4(o[4 * q4] + lo4.x, o[4 * q4 + 1] + lo4.y, o[4 * q4 + 2] + lo4.z,
                                   o[4 * q4 + 3] + lo4.w);
            if (pieces > 1) {
              reinterpret_cast<float4*>(res + 4)[j4] = v;
            } else {
              v.x *= li; v.y *= li; v.z *= li; v.w *= li;
              reinterpret_cast<float4*>(outp)[j4] = v;
            }
          }
        }
        tc_fence_before();
      }
      // every thread is done with the low rows before any writes the next P
      // over them (the two head halves' rows interleave in the buffer)
      soft_bar();
      if (pieces > 1) {
        // the last CTA of the segment merges the partials in CTA order
        __threadfence();
        soft_bar();
        if (threadIdx.x == 0) *s_last = atomicAdd(&a.counters[x.seg], 1u) == (uint32_t)(pieces - 1);
        soft_bar();
        if (*s_last) {
          __threadfence();
          const size_t pstride = (size_t)kAtG * kAtPart;
          const float* ps = a.part + (size_t)x.seg * a.max_pieces * pstride;
          // thread: 128 / (kAtSoft / 64) output dims of head tid / (kAtSoft / 64);
          // a piece's (m, l) and its partial of them loaded together, then
          // folded into the running (max, sum, O), pieces in CTA order
          constexpr int kTh = kAtSoft / kAtG;              // threads per head
          constexpr int kF4 = kD / 4 / kTh;                // output float4s per thread
          const int hh = threadIdx.x / kTh, f0 = (threadIdx.x % kTh) * kF4;
          const float* pm = ps + (size_t)hh * kAtPart;
          float Mx = -INFINITY, Ls = 0.f;
          float4 O[kF4];
#pragma unroll
          for (int q = 0; q < kF4; ++q) O[q] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
          for (int p = 0; p < pieces; ++p) {
            const float* pp = pm + (size_t)p * pstride;
            const float2 ml = __ldcg(reinterpret_cast<const float2*>(pp));
            float4 v[kF4];
#pragma unroll
            for (int q = 0; q < kF4; ++q) v[q] = __ldcg(reinterpret_cast<const float4*>(pp + 4) + f0 + q);
            if (ml.x != -INFINITY) {
              const float M2 = fmaxf(Mx, ml.x);
              const float wa = Mx == -INFINITY ? 0.f : exp2f(Mx - M2), wb = exp2f(ml.x - M2);
              Ls = Ls * wa + ml.y * wb;
#pragma unroll
              for (int q = 0; q < kF4; ++q) {
                O[q].x = O[q].x * wa + v[q].x * wb; O[q].y = O[q].y * wa + v[q].y * wb;
                O[q].z = O[q].z * wa + v[q].z * wb; O[q].w = O[q].w * wa + v[q].w * wb;
              }
              Mx = M2;
            }
          }
          const float li = Ls > 0.f ? 1.f / Ls : 0.f;
          float4* dst = reinterpret_cast<float4*>(a.out + ((size_t)x.lb * a.n_q + (size_t)x.g * kAtG + hh) * kD) + f0;
#pragma unroll
          for (int q = 0; q < kF4; ++q) dst[q] = make_float4(O[q].x * li, O[q].y * li, O[q].z * li, O[q].w * li);
          soft_bar();
          if (threadIdx.x == 0) a.counters[x.seg] = 0u;
        }
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == kAtWarpMma) {
    tc_fence_after();
    tmem_dealloc<kAtTmemCols>(tmem);
  }
}

static size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

size_t attn_tc_extra_bytes(int n_layers, int B, int n_kv, int budget) {
  int nt, tpc, grid, mp;
  attn_tc_plan(n_layers, B, n_kv, budget, &nt, &tpc, &grid, &mp);
  const size_t nseg = (size_t)n_layers * B * n_kv;
  const size_t parts = mp > 1 ? nseg * mp * (size_t)kAtG * kAtPart * sizeof(float) : 0;
  return round256(parts) + (size_t)grid * 8 * kAtMapBytes;
}

int attn_tc_launch(AttnTcCall c, int n_layers, void* stream) {
  int grid;
  attn_tc_plan(n_layers, c.B, c.n_kv, c.K, &c.nt, &c.tpc, &grid, &c.max_pieces, &c.split_pos);
  c.total = n_layers * c.B * c.n_kv * c.nt;
  if (grid < 1) return SPC_OK;
  const size_t nseg = (size_t)n_layers * c.B * c.n_kv;
  const size_t parts = c.max_pieces > 1 ? nseg * c.max_pieces * (size_t)kAtG * kAtPart * sizeof(float) : 0;
  c.maps = reinterpret_cast<uint8_t*>(c.part) + round256(parts);
  // the template of the per-view maps (K or V rows of one KV head: [rows][128]
  // bf16, boxes of 128 rows x 64 dims; base and row count are patched on the
  // device) and the map of the queries ([n_layers B n_q][128], 64-row boxes)
  CUtensorMap tile_tmpl, row_tmpl;
  const uint64_t tdims[2] = {(uint64_t)kD, (uint64_t)kAtRows};
  const uint64_t strides[1] = {(uint64_t)kRowBytes};
  const uint32_t tbox[2] = {64, (uint32_t)kAtRows};
  const uint32_t rbox[2] = {64, 1};
  if (!tensor_map_bf16_sw128(&tile_tmpl, c.q, 2, tdims, strides, tbox) ||
      !tensor_map_bf16_sw128(&row_tmpl, c.q, 2, tdims, strides, rbox))
    return SPC_ERR_CUDA;
  cudaError_t e = set_func_attr((const void*)attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kAtSmem);
  if (e != cudaSuccess) return SPC_ERR_CUDA;
  attn_tc_kernel<<<grid, kAtThreads, kAtSmem, static_cast<cudaStream_t>(stream)>>>(tile_tmpl, row_tmpl, c);
  return cudaGetLastError() == cudaSuccess ? SPC_OK : SPC_ERR_CUDA;
}

}  // namespace spc
