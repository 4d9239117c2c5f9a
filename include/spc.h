/*
 * spc.h -- C ABI of the SpeContext decode-step hot path on GB300 (sm_103a).
 *
 * The method (pages cited by title and section):
 *   [Blog]    "ASPLOS'26 | SpeContext 让小模型先圈出重要 KV Cache" (marsggbo blog)
 *   [Summary] "SpeContext: Enabling Efficient Long-context Reasoning with
 *             Speculative Context Sparsity in LLMs" (paperlayer.ai summary of
 *             arXiv 2512.00722v1)
 *   [SparseSpec-L] news post on SparseSpec-L (only its "sinks + recent window
 *             + top-K" retained set is used here)
 *
 * One decode step, per [Blog] §4: the lightweight retrieval head scores the
 * whole context and selects positions for the NEXT step (spc_score_select);
 * only positions not already resident are loaded (spc_elastic_diff, then
 * spc_gather_kv on a second stream); the LLM attends over the sparse KV that
 * the previous step prepared (spc_sparse_decode_attn).
 *
 * Conventions shared by every call:
 *   - All tensors are row-major, contiguous, and live in device memory unless
 *     a comment says otherwise. bf16 values are bfloat16 bit patterns
 *     (uint16). d (head dimension) must be 128.
 *   - The caller owns every buffer. The library never allocates or frees
 *     memory and keeps no per-call state: scratch space comes from the
 *     caller's workspace.
 *   - Calls are asynchronous on `stream` (a cudaStream_t, NULL = legacy
 *     default stream). Arguments are validated on the host before anything is
 *     launched; a rejected call launches nothing and returns a negative code.
 *   - Returns SPC_OK or a negative spc_status. An error raised by a kernel
 *     after launch surfaces at the caller's next synchronisation (CUDA error)
 *     or in the workspace status word (spc_score_select, spc_sparse_decode_attn,
 *     spc_mla_decode_attn): every bounded device-side wait that gives up
 *     records SPC_ERR_TIMEOUT there, lets its copies in flight land and
 *     returns, so the context stays usable.
 *   - Calls on the same stream may be captured into a CUDA graph once each
 *     entry point has been called once outside capture (the first call sets
 *     kernel attributes).
 */
#ifndef SPC_H_
#define SPC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum spc_status {
  SPC_OK = 0,
  SPC_ERR_INVALID_ARG = -1, /* null or misaligned pointer, bad flag          */
  SPC_ERR_SHAPE = -2,       /* unsupported or inconsistent sizes            */
  SPC_ERR_CUDA = -3,        /* a CUDA runtime call or a launch failed        */
  SPC_ERR_TIMEOUT = -4,     /* a device-side wait gave up (status word only) */
  SPC_ERR_WORKSPACE = -5,   /* workspace missing or too small                */
  SPC_ERR_OVERFLOW = -6     /* appending would exceed the capacity (status)  */
} spc_status;

/* Limits checked on the host. */
#define SPC_HEAD_DIM 128
#define SPC_MAX_CAP 262144      /* positions per request                      */
#define SPC_MAX_BUDGET 4096     /* KV budget per KV head                       */
#define SPC_MAX_BATCH 64
#define SPC_MAX_GROUP 64        /* query heads per KV head (1,2,4,8,16,32,64) */
#define SPC_MAX_HIDDEN 32768    /* retrieval-head input width H               */

/* Human-readable name of a status code. Never NULL. */
const char* spc_status_string(int status);

/* Library version as 10000*major + 100*minor + patch. */
int spc_version(void);

/* ------------------------------------------------------------------------
 * Retrieval head: projection, per-head softmax over the context, GQA group
 * max, forced set + Top-K.
 *   [Blog] §5 (C1): the head keeps the embedding and the Q/K projections and
 *   computes attention weights; selection is per head; for GQA the weights of
 *   a group's query heads are combined by an element-wise max and Top-K is
 *   taken per group; MQA is one group. [Summary] §4.3 (same, "attention
 *   weights"). [Blog] §2: softmax(QK^T/sqrt(d)); the KV budget K is the number
 *   of positions kept per head per step. Sinks and recent window:
 *   [SparseSpec-L], [Summary] §2.2 (StreamingLLM's initial tokens + window).
 *
 * Computes, for every request b and KV head g (G = n_q / n_kv):
 *   q[b,h,:]   = x_b . Wq[:, h*d:(h+1)*d]                     (fp32, unrounded)
 *   if append and len[b] < cap:
 *     K_dlm[b,g,len[b],:] = bf16_rne(x_b . Wk[:, g*d:(g+1)*d]);  len[b] += 1
 *   P_h[p]     = softmax_p(q[b,h] . K_dlm[b,g(h),p] / sqrt(d)),  p < len[b]
 *   s_g[p]     = max_{h in g} P_h[p]
 *   selected[b,g,:] = all p < len (if len <= budget), else
 *                     F U top_{budget-|F|}{ s_g[p] : p not in F },
 *                     F = {0..n_sink-1} U {len-n_recent..len-1};
 *                     ties go to the lower position; ascending; -1 padded.
 *
 * x          bf16 [B][H] head input of this step.
 * Wq         bf16 [H][n_q*d]; Wk bf16 [H][n_kv*d] (may be NULL if !append).
 * K_dlm      bf16 [B][n_kv][cap][d] key cache of the retrieval head, 16-byte
 *            aligned; row len[b] of every head is written when appending.
 * len        int32 [B] context lengths, device memory; read at the start,
 *            incremented by one per request when appending (after every
 *            kernel of this call has read it).
 * q_out      optional fp32 [B][n_q][d] projected queries (NULL: not written).
 * scores_out optional fp32 [B][n_kv][cap]: s_g[p] for p < len (NULL: not
 *            written; entries p >= len are left untouched).
 * selected   int32 [B][n_kv][budget] output.
 * workspace  device scratch of at least spc_score_select_workspace_size()
 *            bytes, 256-byte aligned, ZERO-FILLED BEFORE ITS FIRST USE; every
 *            call leaves it ready for the next one. Its first int32 is the
 *            device status word: 0, or SPC_ERR_TIMEOUT / SPC_ERR_OVERFLOW set
 *            by a kernel; the caller reads and clears it.
 * Limits: d = 128; n_q % n_kv == 0 with G in {1,2,4,8,16,32,64}; H % 8 == 0,
 *         8 <= H <= 32768; 1 <= B <= 64; 1 <= budget <= min(cap, 4096); cap <= 262144;
 *         n_sink + n_recent <= budget.
 * Concurrent calls must use distinct workspaces.
 * ---------------------------------------------------------------------- */
size_t spc_score_select_workspace_size(int B, int H, int n_q, int n_kv, int d, int cap,
                                       int budget);

int spc_score_select(const void* x, const void* Wq, const void* Wk, void* K_dlm, int32_t* len,
                     int append, int B, int H, int n_q, int n_kv, int d, int cap, int budget,
                     int n_sink, int n_recent, float* q_out, float* scores_out,
                     int32_t* selected, void* workspace, size_t workspace_bytes, void* stream);

/* The same call restricted to some of its three kernels, run in order:
 * SPC_STAGE_PROJECT (projection and append), SPC_STAGE_SCAN (key scan and
 * per-head logsumexp partials), SPC_STAGE_SELECT (group score, Top-K, len
 * update). Calling the stages one by one on one stream with one workspace
 * gives the same result as spc_score_select; used to time each kernel. */
#define SPC_STAGE_PROJECT 1
#define SPC_STAGE_SCAN 2
#define SPC_STAGE_SELECT 4
int spc_score_select_stages(const void* x, const void* Wq, const void* Wk, void* K_dlm, int32_t* len,
                            int append, int B, int H, int n_q, int n_kv, int d, int cap, int budget,
                            int n_sink, int n_recent, float* q_out, float* scores_out,
                            int32_t* selected, void* workspace, size_t workspace_bytes,
                            void* stream, int stages);

/* ------------------------------------------------------------------------
 * Elastic loading: the set difference between the new selection and the
 * resident slots. [Blog] §6 (C2): to_load = S_now - S_last, worked example
 * S_last={1,8,21,35}, S_now={1,8,21,50} -> {50}; [Summary] §5.4: reuse the
 * resident entries, fetch only the absent ones, in place under a fixed budget.
 *
 * Per (b, g), with S = {selected[b,g,i] >= 0} and slot s holding
 * slot_pos_prev[b,g,s] (-1 = empty):
 *   kept  = slots whose position is in S (their position is unchanged);
 *   free  = all other slots, ascending slot index;
 *   loads = S minus the kept positions, in the order they appear in
 *           `selected` (ascending positions for spc_score_select's output);
 *   load i goes to free slot i: load_slot[i], load_pos[i], i < n_load[b,g];
 *   slot_pos_next = slot_pos_prev with each free slot set to its load, or -1.
 *
 * selected       int32 [B][n_kv][budget]; distinct positions or -1; positions
 *                outside [0, cap) are ignored.
 * slot_pos_prev  int32 [B][n_kv][budget]; distinct positions or -1.
 * slot_pos_next  int32 [B][n_kv][budget] output; may alias slot_pos_prev.
 * load_slot, load_pos int32 [B][n_kv][budget] outputs (entries >= n_load are
 *                not written); n_load int32 [B][n_kv] output.
 * A second call with the same selection and the new slot map yields n_load = 0.
 * Limits: budget <= 4096, cap <= 262144.
 * ---------------------------------------------------------------------- */
int spc_elastic_diff(const int32_t* selected, const int32_t* slot_pos_prev,
                     int32_t* slot_pos_next, int32_t* load_slot, int32_t* load_pos,
                     int32_t* n_load, int B, int n_kv, int budget, int cap, void* stream);

/* ------------------------------------------------------------------------
 * Gather of the missing K/V rows from pinned host memory into the resident
 * slots, in place, by a kernel that reads host memory directly (no copy
 * engine). [Blog] §4 (asynchronous prefetcher on another CUDA stream), §7
 * (an offloaded layer keeps a budget-sized workspace in GPU memory);
 * [Summary] §5.1 (prefetch concurrent with compute), §5.4 (in place).
 *
 * For model layers l in [layer_lo, layer_hi) held in host memory by request b
 * (view.layer0 <= l < view.layer0 + view.n_layers), for kv in {K, V}, KV head
 * g and i < n_load[b,g], with p = load_pos[b,g,i] and s = load_slot[b,g,i]:
 *   slots[l - view.layer0, kv, g, s, :] = host[p, g, l - view.store_layer0, kv, :]
 * Each row is d bf16 (256 bytes), copied bit-exact.
 *
 * views      device array [B] of spc_gather_view.
 * host       device-visible address of mapped pinned host memory (see
 *            spc_host_device_pointer), POSITION-MAJOR:
 *            bf16 [cap][n_kv][view.store_layers][2][d], 16-byte aligned. One
 *            (position, KV head) holds every stored layer's K and V row
 *            contiguously, so a load reads one run of 512 bytes per layer
 *            from a single host page: the GPU translates host addresses page
 *            by page over the link, and a layer-major store made every
 *            scattered row a separate page (measured: 13-22 GB/s once a step
 *            touched ~100 000 pages of a 64 GiB store, against ~180 GB/s).
 *            store_layer0 is the model layer of the store's layer 0.
 * slots      device memory bf16 [view.n_layers][2][n_kv][budget][d] for layers
 *            [view.layer0, view.layer0 + view.n_layers), 16-byte aligned.
 * The slots being overwritten must not be read concurrently: order this call
 * after the attention that reads the previous contents (an event).
 * Limits: B * n_kv <= 1024, budget <= 4096; the view's host layers must lie
 * inside the store (store_layer0 <= layer0 and layer0 + n_layers <=
 * store_layer0 + store_layers), else the layer is skipped.
 * ---------------------------------------------------------------------- */
typedef struct spc_gather_view {
  const void* host;
  void* slots;
  int32_t layer0;
  int32_t n_layers;
  int32_t store_layer0;
  int32_t store_layers;
} spc_gather_view;

int spc_gather_kv(const spc_gather_view* views, int layer_lo, int layer_hi,
                  const int32_t* load_slot, const int32_t* load_pos, const int32_t* n_load,
                  int B, int n_kv, int d, int cap, int budget, void* stream);

/* ------------------------------------------------------------------------
 * Adaptive memory management (C3). [Blog] §7: thresholds on the sequence
 * length are computed ahead of time from the model's layer count, KV heads and
 * head dimension, the GPU memory available and the number of concurrent
 * requests and the KV budget; each time the context reaches the next
 * threshold the last layer still on the GPU moves its KV to CPU memory and
 * keeps only a budget-sized workspace on the GPU, so GPU memory stays used
 * without a cliff. [Summary] §6.2, §6.2.1 (same, "progressively offloads").
 *
 * spc_offload_thresholds (host only, no GPU needed). With R = 2 * n_kv * d * 2
 * bytes per position and layer (K and V, bf16) and B requests, k offloaded
 * layers at context length s cost B * ((n_layers - k) * s + k * budget) * R
 * bytes of GPU KV memory. For k = 0 .. n_layers-1:
 *   thresholds[k] = floor((kv_bytes / (B * R) - k * budget) / (n_layers - k)) + 1,
 * the shortest length at which k offloaded layers no longer fit, so that at
 * s >= thresholds[k] a (k+1)-th layer must go; thresholds[n_layers] =
 * INT64_MAX. The runtime rule: while s >= thresholds[n_off], offload layer
 * n_layers - 1 - n_off and increment n_off (last layers first).
 * thresholds  host array of n_layers + 1 int64, written on success.
 * Returns SPC_ERR_WORKSPACE when even every layer offloaded (n_layers budget
 * workspaces per request) does not fit in kv_bytes.
 *
 * spc_fill_slots: the workspace of a layer entering CPU memory starts out with
 * the rows the request keeps resident. For layers l in [layer_lo, layer_hi)
 * held by request b's view (view.layer0 <= l < view.layer0 + view.n_layers),
 * kv in {K, V}, KV head g and slot s with 0 <= p = slot_pos[b,g,s] < cap:
 *   view.slots[l', kv, g, s, :] = view.host[l', kv, g, p, :],  l' = l - view.layer0
 * Here view.host is a LAYER-MAJOR cache bf16 [n_layers][2][n_kv][cap][d] (the
 * layer's HBM cache, the usual source; a device-visible host address also
 * works); store_layer0 / store_layers are not used. slots bf16
 * [n_layers][2][n_kv][budget][d]; slot_pos int32 [B][n_kv][budget]. Rows are
 * copied bit-exact. Limits as spc_gather_kv.
 *
 * spc_store_layer: writes one layer's layer-major cache into a position-major
 * host store (the copy half of an offload):
 *   store[p, g, layer, kv, :] = src[kv, g, p, :]   for p < rows, every g, kv,
 * src bf16 [2][n_kv][cap][d] (device memory), store the device-visible address
 * of bf16 [cap][n_kv][store_layers][2][d]; 0 <= layer < store_layers,
 * rows <= cap. A kernel copy (no copy engine), 16-byte aligned addresses.
 * ---------------------------------------------------------------------- */
int spc_offload_thresholds(int n_layers, int n_kv, int d, int B, int budget, int64_t kv_bytes,
                           int64_t* thresholds);

int spc_fill_slots(const spc_gather_view* views, int layer_lo, int layer_hi, const int32_t* slot_pos,
                   int B, int n_kv, int d, int cap, int budget, void* stream);

int spc_store_layer(void* store, const void* src, int n_kv, int d, int cap, int rows, int store_layers,
                    int layer, void* stream);

/* ------------------------------------------------------------------------
 * Sparse GQA decode attention over the resident budget. [Blog] §2 formula
 * over the kept rows; §4: the LLM forward uses the sparse KV prepared in the
 * previous iteration; [Summary] §4.3: for GQA the selected KV serves every
 * query head of its group.
 *
 * For layers l < n_layers, request b, query head h (g = h / G):
 *   rows R = { i : slot_pos[b,g,i] >= 0 }     (view.use_slots = 1: row i of
 *                                              the view is slot i)
 *          = { selected[b,g,i] : >= 0 }       (view.use_slots = 0: positions
 *                                              into a full cache)
 *   out[l,b,h,:] = sum_{r in R} softmax_r(scale * q[l,b,h] . K[g,r]) V[g,r]
 *   (zeros when R is empty).
 *
 * q          bf16 [n_layers][B][n_q][d] LLM queries.
 * views      device array [n_layers][B] of spc_kv_view; k, v point at
 *            bf16 [n_kv][rows][d], 16-byte aligned.
 * selected, slot_pos int32 [B][n_kv][budget] (shared by all layers).
 * out        fp32 [n_layers][B][n_q][d].
 * workspace  device scratch of spc_sparse_decode_attn_workspace_size() bytes
 *            for this call's shapes (the size is not monotone in n_layers: a
 *            caller that launches several layer counts sizes it for each),
 *            256-byte aligned, ZERO-FILLED BEFORE ITS FIRST USE (calls leave
 *            it ready). Its first int32 is the device status word: 0, or
 *            SPC_ERR_TIMEOUT when a bounded wait of the kernel gave up (the
 *            output of that call is then incomplete); the caller reads and
 *            clears it.
 * Limits: d = 128, G in {1,2,4,8,16,32,64}, 1 <= B <= 64, n_layers * B <=
 * 65535, budget <= 4096, scale > 0.
 * G = 64 runs on the tcgen05 tensor cores with TMA loads (K and V of slot
 * views as tiles of contiguous rows, positions as row gathers); the view's
 * k and v then also need 16-byte aligned rows (d = 128 bf16: always).
 * ---------------------------------------------------------------------- */
typedef struct spc_kv_view {
  const void* k;
  const void* v;
  int64_t rows;
  int32_t use_slots;
  int32_t reserved;
} spc_kv_view;

size_t spc_sparse_decode_attn_workspace_size(int n_layers, int B, int n_q, int n_kv, int d,
                                             int budget);

int spc_sparse_decode_attn(const void* q, const spc_kv_view* views, const int32_t* selected,
                           const int32_t* slot_pos, int n_layers, int B, int n_q, int n_kv,
                           int d, int budget, float scale, float* out, void* workspace,
                           size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * spc_sparse_decode_attn without a caller workspace. The paper has no
 * counterpart: this exists for callers that cannot allocate device memory --
 * for example code running under another framework's memory manager, which
 * reserves the device memory up front so a private cudaMalloc would fail or
 * escape its accounting, or a decode loop that must not pay for cudaMalloc /
 * cudaFree and the device-wide synchronisation they can bring.
 *
 * Same arguments, computation and limits as spc_sparse_decode_attn, minus the
 * workspace. Its scratch (split partials and merge counters) lives in a fixed
 * SPC_ATTN_NOALLOC_SCRATCH_BYTES area of the library's own device memory,
 * which every GPU that loads the library holds until the process exits; the
 * call itself allocates nothing. Shapes whose scratch would not fit return
 * SPC_ERR_WORKSPACE before anything is launched (spc_sparse_decode_attn_
 * workspace_size() tells the need). The first call on each device looks up the
 * area's address with that device current; make that first call before any
 * stream capture. Every call clears the status word and the counters it needs
 * (one memset on `stream`) and then launches the kernel. The status word lives
 * in the library's area, which the caller cannot read: a bounded wait that
 * gives up still ends the kernel (the output is then incomplete), but this
 * variant does not report it -- use spc_sparse_decode_attn where that must be
 * observed. All calls share the one area: calls
 * whose work overlaps on the GPU (different streams, or different host
 * threads without ordering) race on it and give wrong results; order them on
 * one stream.
 * ---------------------------------------------------------------------- */
#define SPC_ATTN_NOALLOC_SCRATCH_BYTES (8u << 20)

int spc_sparse_decode_attn_noalloc(const void* q, const spc_kv_view* views,
                                   const int32_t* selected, const int32_t* slot_pos, int n_layers,
                                   int B, int n_q, int n_kv, int d, int budget, float scale,
                                   float* out, void* stream);

/* ------------------------------------------------------------------------
 * Batch-level selection: the alternative the pages compare head-level
 * retrieval with ([Blog] §5: merging every head's weights into one Top-K is
 * too coarse; head-level keeps a set per head). For every request b:
 *   s_b[p] = max_g scores[b,g,p],  p < len[b]
 *   selected[b,g,:] = the spc_score_select rule (forced sinks and recent
 *                     window, Top-K of s_b, ties to the lower position,
 *                     ascending, -1 padded), the SAME set for every KV head g.
 * scores     fp32 [B][n_kv][cap]: the group scores spc_score_select writes to
 *            scores_out in the same step (entries p >= len are not read).
 * len        int32 [B] current lengths (read only).
 * selected   int32 [B][n_kv][budget] output.
 * workspace  spc_batch_select_workspace_size() bytes, 256-byte aligned,
 *            ZERO-FILLED BEFORE ITS FIRST USE (calls leave it ready).
 * Limits: as spc_score_select (B <= 64, budget <= min(cap, 4096), cap <=
 *         262144, n_sink + n_recent <= budget), n_kv <= 64.
 * ---------------------------------------------------------------------- */
size_t spc_batch_select_workspace_size(int B, int cap, int budget);

int spc_batch_select(const float* scores, int32_t* len, int B, int n_kv, int cap, int budget, int n_sink,
                     int n_recent, int32_t* selected, void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * MLA variant. [Blog] §5: for DeepSeek's MLA the retrieval picks entries of
 * the low-dimensional latent cache and only the selected entries are
 * up-projected; [Summary] §4.3: retrieval stays head-level and only the
 * selected latent entries are expanded for attention.
 *
 * Shapes (DeepSeek-V2 style MLA): each position caches ONE latent row of
 * SPC_MLA_LATENT + SPC_MLA_ROPE = 576 bf16 -- a 512-value latent c shared by
 * every head, then a 64-value decoupled rope key. Head h expands c into the
 * key [W_uk[h] c ; c_rope] (128 + 64 values) and the value W_uv[h] c (128);
 * queries carry 128 "nope" values then 64 rope values per head. No RoPE
 * rotation is applied (as in the GQA path). SPC_MLA_HEADS = 16 query heads
 * (DeepSeek-V2-Lite, or one tensor-parallel shard of 8 of DeepSeek-V3's 128).
 * The latent row is shared by all heads, so the 16 heads form one group (as
 * for MQA): one selection per request, n_kv = 1 in the diff and slot maps.
 * ---------------------------------------------------------------------- */
#define SPC_MLA_LATENT 512
#define SPC_MLA_ROPE 64
#define SPC_MLA_NOPE 128
#define SPC_MLA_V 128
#define SPC_MLA_HEADS 16

/* Retrieval head over the latent cache. For every request b:
 *   q[b,h,:]  = x_b . Wq[:, h*192:(h+1)*192]                     (fp32)
 *   if append and len[b] < cap:
 *     C_dlm[b, len[b], :] = bf16_rne(x_b . Wdkv);  len[b] += 1
 *   key_h(p)  = [Wuk[h] C_dlm[b,p,:512] ; C_dlm[b,p,512:]]
 *   P_h[p]    = softmax_p(q[b,h] . key_h(p) / sqrt(192)),  p < len[b]
 *   s[p]      = max_h P_h[p]
 *   selected[b,:] = as spc_score_select with one group (forced sinks and
 *               recent window, Top-K, ties to the lower position, -1 padded).
 * Computed with the query absorbed into the latent space,
 * [Wuk[h]^T q_nope ; q_rope] . C_dlm[b,p], the same quantity.
 *
 * x          bf16 [B][H].
 * Wq         bf16 [H][16*192].
 * Wuk        bf16 [16][128][512]: row j of head h maps the latent to key value j.
 * Wdkv       bf16 [H][576] latent down-projection (may be NULL if !append).
 * C_dlm      bf16 [B][cap][576] latent cache of the retrieval head, 16-byte
 *            aligned; row len[b] is written when appending.
 * len, scores_out ([B][cap]), selected ([B][budget]), workspace, status word
 *            and stages: as spc_score_select_stages (the workspace size from
 *            spc_mla_score_select_workspace_size). The projection stage also
 *            absorbs the queries.
 * Limits: H % 8 == 0, 8 <= H <= 32768; 1 <= B <= 64; 1 <= budget <=
 *         min(cap, 4096); cap <= 262144; n_sink + n_recent <= budget.
 * ---------------------------------------------------------------------- */
size_t spc_mla_score_select_workspace_size(int B, int H, int cap, int budget);

int spc_mla_score_select(const void* x, const void* Wq, const void* Wuk, const void* Wdkv, void* C_dlm,
                         int32_t* len, int append, int B, int H, int cap, int budget, int n_sink,
                         int n_recent, float* scores_out, int32_t* selected, void* workspace,
                         size_t workspace_bytes, void* stream, int stages);

/* Gather of missing latent rows from pinned host memory (spc_gather_kv with
 * one KV head and 576-value rows, no K/V pair). For host layers l of request
 * b and load i < n_load[b], p = load_pos[b,i], s = load_slot[b,i]:
 *   slots[l - view.layer0, s, :] = host[p, l - view.store_layer0, :]
 * host   POSITION-MAJOR bf16 [cap][view.store_layers][576] (one position's
 *        latent rows of every stored layer are contiguous), device-visible
 *        address of mapped pinned memory, 16-byte aligned.
 * slots  bf16 [view.n_layers][budget][576] device memory, 16-byte aligned.
 * load_slot, load_pos int32 [B][budget], n_load int32 [B] (spc_elastic_diff
 * with n_kv = 1). Order after the attention that reads the old slot rows.
 * Limits: 1 <= B <= 64, budget <= 4096, cap <= 262144; the view's host
 * layers must lie inside the store, else the layer is skipped. */
int spc_mla_gather(const spc_gather_view* views, int layer_lo, int layer_hi, const int32_t* load_slot,
                   const int32_t* load_pos, const int32_t* n_load, int B, int cap, int budget,
                   void* stream);

/* Sparse MLA decode attention over the selected latent rows, for n_layers
 * layers x B requests (unit u = layer * B + b):
 *   out[u,h,:] = sum_r softmax_r(q[u,h] . key_{l,h}(C_r) * scale) W_uv[l,h] C_r[:512]
 * over the rows r the view keeps (as spc_sparse_decode_attn: positions of
 * `selected` into a full cache, or slots with slot_pos >= 0), with
 * key_{l,h}(c) = [W_uk[l,h] c[:512] ; c[512:]]. Computed with the query
 * absorbed and W_uv applied once to the softmax-weighted latent sum (the same
 * quantity as up-projecting every selected row).
 * q          bf16 [n_layers][B][16][192] LLM queries (nope, then rope values).
 * Wuk, Wuv   bf16 [n_layers][16][128][512].
 * views      device array [n_layers][B] of spc_kv_view: k = latent rows bf16
 *            [rows][576] (16-byte aligned), v unused (NULL), rows, use_slots.
 * selected, slot_pos int32 [B][budget] (shared by all layers).
 * out        fp32 [n_layers][B][16][128].
 * workspace  device scratch of spc_mla_decode_attn_workspace_size() bytes,
 *            256-byte aligned; its first int32 is a status word (0, or
 *            SPC_ERR_TIMEOUT set by a kernel), ZERO-FILLED BEFORE FIRST USE.
 * Limits: 1 <= B <= 64, budget <= 4096, n_layers * B <= 65535, scale > 0;
 * q, Wuk, Wuv and out 16-byte aligned. */
size_t spc_mla_decode_attn_workspace_size(int n_layers, int B, int budget);

int spc_mla_decode_attn(const void* q, const void* Wuk, const void* Wuv, const spc_kv_view* views,
                        const int32_t* selected, const int32_t* slot_pos, int n_layers, int B, int budget,
                        float scale, float* out, void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Helpers (no counterpart on the pages).
 * ---------------------------------------------------------------------- */

/* Device-visible address of pinned host memory allocated with
 * cudaHostAlloc/cudaMallocHost or registered with cudaHostRegister
 * (cudaHostGetDevicePointer). Returns SPC_ERR_CUDA for other memory. */
int spc_host_device_pointer(void* host_ptr, void** device_ptr);

/* Streams `bytes` (a multiple of 16) from `src` (device memory or a
 * device-visible host address) with 16-byte loads over `n_blocks` CTAs of 512
 * threads, folding the data into sink[blockIdx] so no load is dropped. Used to
 * measure the HBM and host-link read bandwidth the kernels are compared with.
 * sink: uint32 [n_blocks]. src 16-byte aligned. */
int spc_stream_read(const void* src, size_t bytes, uint32_t* sink, int n_blocks, void* stream);

/* Copies `bytes` from `src` to `dst` with a kernel (no copy engine): either
 * address may be device memory or the device-visible address of mapped
 * pinned host memory (spc_host_device_pointer). The pages have no
 * counterpart; it is the host I/O of a decode loop captured in a CUDA graph,
 * where a copy-engine transfer to or from host memory inside the graph stalled
 * every step, while this kernel reads and writes the mapped memory directly.
 * 16-byte aligned addresses move in 16-byte words; any other bytes move one
 * at a time. Up to 16 CTAs of 256 threads, so it leaves the GPU to the other
 * streams. src and dst must not overlap. */
int spc_copy(void* dst, const void* src, size_t bytes, void* stream);

/* Number of streaming multiprocessors of the current device (0 on error). */
int spc_device_sm_count(void);

#ifdef __cplusplus
}
#endif
#endif /* SPC_H_ */
