// Host-side declarations shared by the translation units of libspc.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "spc.h"

namespace spc {

// Sets a kernel attribute on the current device unless a value at least as
// large is already set there (dynamic shared memory size, or a 0/1 flag).
// Kernel attributes belong to a device's context, so the record is kept per
// (kernel, attribute, device); safe to call from several host threads.
cudaError_t set_func_attr(const void* fn, cudaFuncAttribute attr, int value);

struct ScoreSelectCall {
  const void* x;
  const void* Wq;
  const void* Wk;
  void* K_dlm;
  int32_t* len;
  int append;
  int B, H, n_q, n_kv, cap, budget, n_sink, n_recent;
  float* q_out;
  float* scores_out;
  int32_t* selected;
  void* workspace;
  void* stream;
  int stages;
};

size_t score_select_workspace(int B, int H, int n_q, int n_kv, int cap);

// A tiled TMA tensor map of a bf16 tensor with the 128-byte swizzle: `rank`
// dimensions (innermost first), byte strides of dimensions 1 .. rank - 1,
// the box to copy. Encoded through the driver entry point of
// cuTensorMapEncodeTiled (looked up once); false when that fails.
bool tensor_map_bf16_sw128(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                           const uint64_t* strides, const uint32_t* box);

// Retrieval head for groups of 16, 32 or 64 query heads on the 5th-generation
// tensor cores (scan_tc.cu), in two passes over the key cache:
// scan_tc_launch writes scan_tc_ppt(G) logsumexp partials per (head,
// 128-position tile) into `part`; scan_tc_scores_launch folds them into
// `lse` [B][n_q] (base 2), writes the log2 group score of every position into
// `gscore` [B * n_kv][lstride], and the partials of a zero normaliser (one
// per tile) into part1 [B * n_kv][n_parts1] for the radix select.
struct ScanTcCall {
  const uint16_t* K;
  const float* q;
  const int32_t* len;
  float2* part;
  float* lse;
  float* gscore;
  int* status;
  int B, n_q, n_kv, cap, lstride, n_tiles, total_tiles, append, n_parts;
  float qscale;
};
int scan_tc_ppt(int G);
int scan_tc_launch(ScanTcCall c, int G, void* stream);
int scan_tc_scores_launch(ScanTcCall c, int G, float2* part1, int n_parts1, void* stream);

// Sparse decode attention of groups of 64 query heads (attn_tc.cu, tcgen05):
// the arguments of spc_sparse_decode_attn with the workspace split into the
// status word, one merge counter per (layer, request, KV head), and then
// attn_tc_extra_bytes of split partials and per-CTA tensor maps (from
// `part` on, 256-byte aligned). attn_tc_launch fills the tiling fields (nt,
// tpc, total, max_pieces, split_pos) and `maps`.
struct AttnTcCall {
  const uint16_t* q;
  const spc_kv_view* views;
  const int32_t* selected;
  const int32_t* slot_pos;
  float* out;
  float* part;
  uint8_t* maps;
  uint32_t* counters;
  int* status;
  int B, n_q, n_kv, K;
  int nt, tpc, total, max_pieces;
  int split_pos;   // one segment per CTA, position-read segments over two CTAs
  float scale2;
  long long wait_limit;
  int starve;
};
int attn_tc_group();
size_t attn_tc_extra_bytes(int n_layers, int B, int n_kv, int budget);
int attn_tc_launch(AttnTcCall c, int n_layers, void* stream);
int score_select_launch(const ScoreSelectCall& c);

int elastic_diff_launch(const int32_t* selected, const int32_t* prev, int32_t* next,
                        int32_t* load_slot, int32_t* load_pos, int32_t* n_load, int B, int n_kv,
                        int budget, int cap, void* stream);

int gather_launch(const spc_gather_view* views, int layer_lo, int layer_hi, const int32_t* load_slot,
                  const int32_t* load_pos, const int32_t* n_load, int B, int n_kv, int cap,
                  int budget, void* stream);

int fill_slots_launch(const spc_gather_view* views, int layer_lo, int layer_hi, const int32_t* slot_pos,
                      int B, int n_kv, int cap, int budget, void* stream);

int store_layer_launch(void* store, const void* src, int n_kv, int cap, int rows, int store_layers, int layer,
                       void* stream);

size_t attn_workspace(int n_layers, int B, int n_q, int n_kv, int budget);
int attn_launch(const void* q, const spc_kv_view* views, const int32_t* selected,
                const int32_t* slot_pos, int n_layers, int B, int n_q, int n_kv, int budget,
                float scale, float* out, void* workspace, void* stream);

int attn_noalloc_launch(const void* q, const spc_kv_view* views, const int32_t* selected,
                        const int32_t* slot_pos, int n_layers, int B, int n_q, int n_kv, int budget,
                        float scale, float* out, void* stream);

struct MlaScoreSelectCall {
  const void* x;
  const void* Wq;
  const void* Wuk;
  const void* Wdkv;
  void* C_dlm;
  int32_t* len;
  int append;
  int B, H, cap, budget, n_sink, n_recent;
  float* scores_out;
  int32_t* selected;
  void* workspace;
  void* stream;
  int stages;
};

size_t mla_score_select_workspace(int B, int cap);
int mla_score_select_launch(const MlaScoreSelectCall& c);
int mla_absorb_launch(const void* q, int q_bf16, const void* Wuk, int n_items, int items_per_w, float* qa,
                      void* stream);
size_t mla_attn_workspace(int n_layers, int B, int budget);
int mla_attn_launch(const void* q, const void* Wuk, const void* Wuv, const spc_kv_view* views,
                    const int32_t* selected, const int32_t* slot_pos, int n_layers, int B, int budget,
                    float scale, float* out, void* workspace, void* stream);
int mla_gather_launch(const spc_gather_view* views, int layer_lo, int layer_hi, const int32_t* load_slot,
                      const int32_t* load_pos, const int32_t* n_load, int B, int budget, void* stream);

size_t batch_select_workspace(int B, int cap, int budget);
int batch_select_launch(const float* scores, int32_t* len, int B, int n_kv, int cap, int budget, int n_sink,
                        int n_recent, int32_t* selected, void* workspace, void* stream);

int stream_read_launch(const void* src, size_t bytes, uint32_t* sink, int n_blocks, void* stream);

int device_sm_count();

}  // namespace spc
