// Elastic loading: set difference between the new selection and the resident
// KV slots, with the in-place slot assignment.
//
// Method: "ASPLOS'26 | SpeContext 让小模型先圈出重要 KV Cache" (marsggbo blog)
// §6 (C2): to_load = S_now - S_last (worked example {1,8,21,35} ->
// {1,8,21,50} loads {50} into the slot that held 35); "SpeContext: Enabling
// Efficient Long-context Reasoning with Speculative Context Sparsity in LLMs"
// (paperlayer.ai summary) §5.4: reuse what is resident, fetch only the absent
// entries, in place under a fixed budget.
//
// One CTA per (request, KV head). A bitmap of the context (cap bits, at most
// 32 KiB) in shared memory marks the new selection; every resident slot tests
// and clears its bit (kept), so the bits left set are exactly the positions
// to load. Two block-wide ordered scans give the rank of every load (in
// selection order) and of every free slot (in slot order); load i goes to
// free slot i.
#include "spc_device.cuh"
#include "spc_internal.h"

namespace spc {

constexpr int kDiffThreads = 1024;

__global__ void __launch_bounds__(kDiffThreads)
diff_kernel(const int32_t* __restrict__ selected, const int32_t* prev, int32_t* next,
            int32_t* __restrict__ load_slot, int32_t* __restrict__ load_pos,
            int32_t* __restrict__ n_load, int K, int cap) {
  extern __shared__ uint32_t dsm[];
  __shared__ int scratch[33];
  const int nwords = (cap + 31) >> 5;
  uint32_t* bm = dsm;
  int* lp = reinterpret_cast<int*>(dsm + nwords);  // [K] positions to load, in order
  const size_t base = (size_t)blockIdx.x * K;
  const int tid = threadIdx.x;
  const int per = (K + kDiffThreads - 1) / kDiffThreads;  // <= 4

  for (int i = tid; i < nwords; i += kDiffThreads) bm[i] = 0u;
  __syncthreads();
  for (int i = tid; i < K; i += kDiffThreads) {
    const int p = selected[base + i];
    if (p >= 0 && p < cap) atomicOr(&bm[p >> 5], 1u << (p & 31));
  }
  __syncthreads();

  // slots owned by this thread: [tid*per, tid*per + per); every read of
  // `prev` happens before the first barrier below, so next may alias prev
  int pos[4];
  bool keep[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int s = tid * per + k;
    pos[k] = -1;
    keep[k] = false;
    if (k < per && s < K) {
      pos[k] = prev[base + s];
      keep[k] = pos[k] >= 0 && pos[k] < cap && ((bm[pos[k] >> 5] >> (pos[k] & 31)) & 1u);
    }
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < 4; ++k)
    if (keep[k]) atomicAnd(&bm[pos[k] >> 5], ~(1u << (pos[k] & 31)));
  __syncthreads();

  // positions still marked are the loads; rank them in selection order
  int sp[4];
  int lcount = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = tid * per + k;
    int p = -1;
    if (k < per && i < K) p = selected[base + i];
    const bool ld = p >= 0 && p < cap && ((bm[p >> 5] >> (p & 31)) & 1u);
    sp[k] = ld ? p : -1;
    lcount += ld ? 1 : 0;
  }
  int nl;
  int lr = block_excl_scan(lcount, scratch, &nl);
#pragma unroll
  for (int k = 0; k < 4; ++k)
    if (sp[k] >= 0) lp[lr++] = sp[k];

  int fcount = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int s = tid * per + k;
    fcount += (k < per && s < K && !keep[k]) ? 1 : 0;
  }
  int nf;
  int fr = block_excl_scan(fcount, scratch, &nf);  // its barriers also publish lp

#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int s = tid * per + k;
    if (k >= per || s >= K) continue;
    if (keep[k]) {
      next[base + s] = pos[k];
    } else {
      if (fr < nl) {
        const int p = lp[fr];
        next[base + s] = p;
        load_slot[base + fr] = s;
        load_pos[base + fr] = p;
      } else {
        next[base + s] = -1;
      }
      ++fr;
    }
  }
  if (tid == 0) n_load[blockIdx.x] = nl;
}

int elastic_diff_launch(const int32_t* selected, const int32_t* prev, int32_t* next,
                        int32_t* load_slot, int32_t* load_pos, int32_t* n_load, int B, int n_kv,
                        int budget, int cap, void* stream) {
  const size_t smem = sizeof(uint32_t) * (size_t)((cap + 31) / 32) + sizeof(int) * (size_t)budget;
  if (set_func_attr((const void*)diff_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return SPC_ERR_CUDA;
  diff_kernel<<<B * n_kv, kDiffThreads, smem, static_cast<cudaStream_t>(stream)>>>(
      selected, prev, next, load_slot, load_pos, n_load, budget, cap);
  return cudaGetLastError() == cudaSuccess ? SPC_OK : SPC_ERR_CUDA;
}

}  // namespace spc
