/*
 * pod.h — C ABI of the GB300 (sm_103a) POD paged-attention library.
 *
 * POD ("prefill-on-decode") runs causal prefill attention for one or more
 * requests and batched decode attention for many in-flight requests in ONE
 * kernel launch, both reading a paged KV cache with GQA, and returns outputs
 * plus base-2 LSE for both halves (POD walkthrough, "POD 是什么" and "批量
 * POD：BatchPODWithPagedKVCacheWrapper 完整示例"; run returns
 * ((out_p, lse_p), (out_d, lse_d)) per "BatchPOD 的 run 差异").
 *
 * Life cycle (POD walkthrough, "plan/run 生命周期"): plan once on the host,
 * run many times (for example once per transformer layer) with the same page
 * tables. Every policy (causal, window_left, sm_scale, sinks on/off, dtype) is
 * fixed at plan time, as the walkthrough's "plan 覆盖" rule does for the decode
 * side ("Decode 侧参数与'plan 覆盖'行为"); run takes tensors only. Optional
 * policies are set on the handle between pod_plan and pod_run:
 * pod_plan_set_decode_fp8, pod_plan_set_kv_layout,
 * pod_plan_set_logits_transform, pod_plan_set_rope,
 * pod_plan_set_prefill_mask and pod_plan_set_graph_capacity (then
 * pod_replan plans each new step into the same workspace).
 *
 * Conventions shared by every entry point
 *  - Errors are returned as pod_status codes; nothing aborts or throws.
 *    pod_last_error() returns a thread-local message for the last failure.
 *  - Index arrays passed to pod_plan are HOST int32 arrays (read during the
 *    call only; the caller keeps ownership). Tensor arguments of pod_run are
 *    DEVICE pointers owned by the caller; the library never frees them.
 *  - The handle (host memory) is owned by the library until pod_destroy.
 *  - `stream` is a cudaStream_t passed as void*; NULL is the legacy stream.
 *
 * Tensor layouts (all row-major, contiguous)
 *  - q_p : [p_q_indptr[p_batch], H, d]    q_d : [d_q_indptr[d_batch], H, d]
 *  - kv_p: [p_num_pages, 2, page_size, Hk, d]   kv_d: [d_num_pages, 2, page_size, Hk, d]
 *    (NHD paged cache, index 0 = K, 1 = V; POD walkthrough single-request
 *    docstring example); per half [num_pages, 2, Hk, page_size, d] (HND)
 *    after pod_plan_set_kv_layout
 *  - out_p / out_d: same shape and dtype as q_p / q_d
 *  - lse_p / lse_d: fp32 [rows, H], base 2 (flashinfer.cudnn page, "LSE 契约")
 *  - sinks: fp32 [H] or NULL (flashinfer.cudnn page, "Decode 能力矩阵与参数")
 *  with H = num_qo_heads, Hk = num_kv_heads, d = head_dim.
 */
#ifndef POD_GB300_H
#define POD_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pod_plan_s* pod_handle;

typedef enum {
    POD_OK = 0,
    POD_ERR_INVALID_ARG = 1,    /* inconsistent page tables, heads, lengths */
    POD_ERR_UNSUPPORTED = 2,    /* head_dim / dtype / group size not built */
    POD_ERR_WORKSPACE = 3,      /* workspace missing or too small */
    POD_ERR_CUDA = 4,           /* a CUDA runtime call failed */
    POD_ERR_DEVICE_STATUS = 5   /* a kernel recorded an error (bounded wait ran out) */
} pod_status;

typedef enum { POD_F16 = 0, POD_BF16 = 1 } pod_dtype;

/*
 * pod_plan — host planner (POD walkthrough, "plan 内部做了什么" and "Batch 版本
 * plan 的 colocated-CTA 调度细节").
 *
 * Validates the two page tables, computes kv_len per request
 * (kv_len = (pages - 1) * page_size + last_page_len), cuts prefill queries
 * into 128-row tiles (GQA heads of one KV head packed into rows), splits
 * decode KV ranges into chunks, assigns the work of both halves to the CTAs
 * of one persistent launch and lays out the workspace.
 *
 * Arguments
 *  p_q_indptr[p_batch+1], p_kv_indptr[p_batch+1], p_kv_indices[p_kv_indptr[p_batch]],
 *  p_last_page_len[p_batch]: prefill page tables (host int32). Same for d_*.
 *  p_batch / d_batch may be 0 (that half is empty; its pointers may be NULL).
 *  p_num_pages / d_num_pages: page-pool sizes; every index must be below them.
 *  causal: bottom-right diagonal mask on both halves; window_left: -1 = off,
 *  else keys strictly before the diagonal that stay visible; sm_scale <= 0
 *  means 1/sqrt(head_dim). dtype: element type of q/kv/out. has_sinks: pod_run
 *  will receive a sinks array. num_sms: SM count the schedule is built for
 *  (0 = the current device's); the plan is a pure function of its inputs and
 *  num_sms.
 *  workspace / workspace_bytes: device buffer the plan metadata is copied into
 *  (one cudaMemcpyAsync on `stream`, the only host-to-device copy of the
 *  library). workspace == NULL plans on the host only: the returned handle can
 *  be inspected (pod_workspace_size, pod_plan_table) and bound later with
 *  pod_bind_workspace. Not capturable in a CUDA graph (POD walkthrough,
 *  "plan/run 生命周期": plan cannot run inside CUDA Graph capture).
 *  required_workspace_bytes (may be NULL): receives the size the plan needs,
 *  also when POD_ERR_WORKSPACE is returned.
 *
 * Errors: POD_ERR_INVALID_ARG when num_qo_heads % num_kv_heads != 0, an indptr
 * is not monotone from 0, last_page_len is outside [1, page_size] for a
 * request with queries, an index is outside the pool, kv_len < q_len under
 * causal, or kv_len == 0 for a request with queries. POD_ERR_UNSUPPORTED for
 * head_dim other than 64/128/256, more than 128 qo heads per KV head, or
 * more than 32 qo heads per KV head on the decode half. At head_dim 256 the
 * fused kernel runs one CTA per SM (its O takes 256 TMEM columns and its
 * prefill stages most of the shared memory); RoPE, FP8 decode caches, the
 * soft cap and ALiBi are not built there (refused by their setters). POD_ERR_WORKSPACE when the
 * workspace is too small. On error *out_handle is NULL.
 */
pod_status pod_plan(const int32_t* p_q_indptr, const int32_t* p_kv_indptr,
                    const int32_t* p_kv_indices, const int32_t* p_last_page_len,
                    int32_t p_batch, int32_t p_num_pages,
                    const int32_t* d_q_indptr, const int32_t* d_kv_indptr,
                    const int32_t* d_kv_indices, const int32_t* d_last_page_len,
                    int32_t d_batch, int32_t d_num_pages,
                    int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                    int32_t page_size, int32_t causal, int32_t window_left,
                    float sm_scale, pod_dtype dtype, int32_t has_sinks, int32_t num_sms,
                    void* workspace, size_t workspace_bytes, void* stream,
                    pod_handle* out_handle, size_t* required_workspace_bytes);

/* Bytes of device workspace the plan needs (0 for a NULL handle). Library
 * mechanics (the pages size the workspace by hand); no passage. */
size_t pod_workspace_size(pod_handle h);

/*
 * pod_bind_workspace — copy a host-only plan's metadata into `workspace`
 * (device, >= pod_workspace_size bytes) on `stream`, and wait for the copy
 * (it reads host memory the handle owns). After it, pod_run may be called
 * with this workspace. Library mechanics (plan on the host first, learn the
 * size, then bind); no passage. Errors: POD_ERR_WORKSPACE, POD_ERR_CUDA.
 */
pod_status pod_bind_workspace(pod_handle h, void* workspace, size_t workspace_bytes, void* stream);

/*
 * pod_run — the fused launch (POD walkthrough, "run 的两次'设置'与一次 launch"
 * and "PDL：让两个任务真正并发").
 *
 * Launches the persistent POD kernel (prefill tiles on tcgen05 tensor cores
 * and split-KV decode on the same grid), then, when the plan split any KV
 * range, the partial-output/LSE merge kernel chained with programmatic
 * dependent launch. With RoPE (pod_plan_set_rope) the rotated-copy pre-pass
 * kernels run first on the same stream. No host synchronisation; capturable
 * in a CUDA graph.
 * q_p/kv_p may be NULL when the prefill half is empty (same for the decode
 * half). lse_p / lse_d may be NULL (LSE not written). sinks must be non-NULL
 * exactly when the plan has has_sinks. `workspace` must be the buffer the
 * plan was bound to; it is read and written (plan metadata, split partials,
 * device status word); calls that share a workspace must not overlap.
 * Errors: POD_ERR_INVALID_ARG (NULL tensor for a non-empty half, sinks
 * mismatch, unbound handle, a custom prefill mask that is not device
 * memory), POD_ERR_CUDA (launch failure).
 */
pod_status pod_run(pod_handle h, const void* q_p, const void* kv_p,
                   const void* q_d, const void* kv_d, const float* sinks,
                   void* workspace, void* out_p, float* lse_p,
                   void* out_d, float* lse_d, void* stream);

/*
 * pod_plan_set_decode_fp8 — the decode half's cache is FP8 E4M3 with
 * per-tensor calibration scales (POD walkthrough, "Decode 侧参数与'plan 覆盖'
 * 行为": q_scale and k_scale multiply the decode sm_scale, v_scale multiplies
 * the decode output). From the next pod_run on, kv_d is read as
 * [d_num_pages, 2, page_size, Hk, head_dim] one-byte E4M3 codes, K = code *
 * k_scale and V = code * v_scale; fold a query scale into k_scale. The
 * kernel folds k_scale into its softmax scale and multiplies the decode
 * outputs (split partials included) by v_scale; the decode LSE is that of the
 * scaled logits. q_d and out_d keep the plan's 16-bit dtype; the prefill half
 * is unchanged. Both products run on e4m3 tensor cores with the codes as
 * they are: each query row enters as e4m3 parts of the row scaled by a power
 * of two, which hold a bf16 row exactly and an fp16 row to 12 significant
 * bits, and the softmax weights as two e4m3 parts (about 8 significant bits
 * for weights above 2^-10 of the row's largest, as the bf16 weights of the
 * 16-bit path, and within about 2^-18 of the largest below). May be called
 * again to change the scales. Errors:
 * POD_ERR_UNSUPPORTED unless head_dim is 128, or with a logits transform set
 * (pod_plan_set_logits_transform) or RoPE (pod_plan_set_rope);
 * POD_ERR_INVALID_ARG for a NULL handle or scales that are not finite and
 * positive.
 */
pod_status pod_plan_set_decode_fp8(pod_handle h, float k_scale, float v_scale);

/*
 * pod_plan_set_logits_transform — a transform of every logit, applied by
 * both halves before masking and softmax (FlashInfer guide, "快速上手":
 * logits_soft_cap and pos_encoding_mode ALIBI; the POD plan keeps them).
 * logits_soft_cap > 0: the scaled logit x = sm_scale * q.k becomes
 *   cap * tanh(x / cap); 0 turns it off.
 * alibi_slopes: DEVICE pointer to H fp32 slopes (caller-owned, read by every
 *   later pod_run) or NULL: the logit of key t for a query at bottom-right
 *   position p gains slope[head] * (t - p).
 * Sinks stay plain logits; the LSE is that of the transformed logits.
 * Takes effect from the next pod_run; the plan and workspace are kept.
 * Errors: POD_ERR_INVALID_ARG (NULL handle, negative or non-finite cap),
 * POD_ERR_UNSUPPORTED (both at once, ALiBi under RoPE, either with an FP8
 * decode cache or at head_dim 256; pod_run also refuses slopes that are not
 * device memory).
 */
pod_status pod_plan_set_logits_transform(pod_handle h, float logits_soft_cap,
                                         const float* alibi_slopes);

/*
 * pod_plan_set_rope — rotary position encoding of both halves (FlashInfer
 * guide, "快速上手": pos_encoding_mode ROPE_LLAMA with rope_scale, default
 * 1, and rope_theta, default 1e4; the POD plan keeps them).
 * Queries and keys are rotated before the dot product: a query row at its
 * bottom-right position p = kv_len - q_len + i, key t at t; element j pairs
 * with j + head_dim/2 and turns by (pos / rope_scale) * rope_theta^(-2j/d).
 * Values are not rotated. rope_scale = 0 turns it off.
 * No rotated operand is rounded to 16 bits: each is kept as a 16-bit high
 * part and a 16-bit low part, and every logit is formed as
 * q_hi.k_hi + q_hi.k_lo + q_lo.k_hi. Each pod_run first writes the rotated
 * queries of both halves, and copies of the prefill half's pages (rotated K
 * as high and low parts, V), into the workspace; the workspace grows by
 * about 1.5x the prefill pages plus twice the queries. Decode keys are
 * rotated inside the fused kernel, read once from the caller's cache. The
 * caller's tensors are only read. Under RoPE the fused kernel runs one CTA
 * per SM (the low parts need the shared memory of a second CTA).
 * Switching it on, off or to other values plans the handle again: any bound
 * workspace is released, bind again (the size changes).
 * Errors: POD_ERR_INVALID_ARG (NULL handle, non-finite or non-positive
 * values), POD_ERR_UNSUPPORTED (with an FP8 decode cache, at head_dim 256,
 * or with ALiBi slopes set: one position encoding at a time).
 */
pod_status pod_plan_set_rope(pod_handle h, float rope_scale, float rope_theta);

/*
 * pod_plan_set_kv_layout — page layout of each half's cache (FlashInfer
 * guide, "快速上手", kv_layout: NHD or HND orders the k/v dimensions; the
 * POD run takes one layout per half).
 * p_layout / d_layout: 0 = NHD, pages [2, page_size, Hk, head_dim] (the
 *   default); 1 = HND, pages [2, Hk, page_size, head_dim]. The page pool is
 *   [num_pages, ...] either way and the page tables are unchanged.
 * Takes effect from the next pod_run; the plan and its workspace are kept.
 * With an FP8 decode cache the same two layouts apply to the one-byte codes.
 * Errors: POD_ERR_INVALID_ARG (NULL handle, a layout other than 0 or 1).
 */
pod_status pod_plan_set_kv_layout(pod_handle h, int32_t p_layout, int32_t d_layout);

/*
 * pod_plan_set_prefill_mask — a custom mask on the prefill half (POD
 * walkthrough, "run 参数详解", prefill parameters: custom_mask_p /
 * packed_custom_mask_p, packed with little bit order; a custom mask takes
 * precedence over causal).
 *
 * packed_mask: DEVICE pointer, caller-owned, read by every later pod_run
 *   until replaced; it must stay valid while those runs execute. It holds
 *   one bit per (query row, key) of every prefill request: request r's
 *   [q_len_r, kv_len_r] matrix in row-major order, the requests end to end,
 *   eight bits to a byte with the first in the least significant bit. A set
 *   bit allows the key. mask_bytes is its size; it must cover
 *   ceil(sum_r q_len_r * kv_len_r / 8) bytes, and no byte past mask_bytes is
 *   read. NULL removes the mask (mask_bytes ignored).
 * Semantics: on the prefill half the mask replaces the causal rule;
 *   window_left still applies; the decode half is unchanged. A row the mask
 *   leaves without keys gets out = 0 and lse = -inf.
 * Switching the mask on or off plans the handle again from its own copies of
 *   the page tables (prefill tiles then span every key the window allows):
 *   any bound workspace is released, so call pod_workspace_size and
 *   pod_bind_workspace again before the next pod_run. Replacing one mask
 *   pointer by another keeps the plan and its workspace.
 * Errors: POD_ERR_INVALID_ARG (NULL handle, mask_bytes too small).
 */
pod_status pod_plan_set_prefill_mask(pod_handle h, const void* packed_mask, int64_t mask_bytes);

/*
 * pod_plan_set_graph_capacity — plans for CUDA-graph replay (POD walkthrough,
 * "CUDAGraph 模式的运行时约束": a fixed batch, page-table buffers reserved at
 * their maximum size, and plan run outside capture).
 *
 * max_p_batch / max_p_rows / max_p_pages: the most prefill requests, query
 * rows and page-table entries any later plan of this handle will have; the
 * same for the decode half. All zero turns the mode off. From then on:
 *  - the workspace layout depends on these capacities only
 *    (pod_workspace_size reports it; bind again, the handle's workspace is
 *    released);
 *  - every launch runs the full grid (two CTAs per SM), the merge kernel is
 *    always launched, and the kernels read the plan's counts from the
 *    workspace, so a pod_run captured once serves every later plan;
 *  - the q and out tensors passed to pod_run hold max_*_rows rows (rows past
 *    the plan's own are neither read for keys nor written), and a half with a
 *    non-zero capacity needs its tensors on every run;
 *  - page sizes below 8 use the cp.async gather (the load path may not
 *    depend on the page tables), and prefill key ranges are not split.
 * Library mechanics beyond the passage (its capacity rules are the pages';
 * the fixed layout is this library's way to meet them).
 * Errors: POD_ERR_INVALID_ARG (NULL handle, a negative capacity, or the
 * current plan exceeding one), POD_ERR_UNSUPPORTED (with RoPE or a custom
 * prefill mask).
 */
pod_status pod_plan_set_graph_capacity(pod_handle h, int32_t max_p_batch, int32_t max_p_rows,
                                       int32_t max_p_pages, int32_t max_d_batch,
                                       int32_t max_d_rows, int32_t max_d_pages);

/*
 * pod_replan — plan new page tables into a capacity handle's bound workspace
 * (POD walkthrough, "CUDAGraph 模式的运行时约束": each step plans again,
 * outside capture, within the reserved sizes; "plan/run 生命周期").
 * The arrays are host int32 as for pod_plan (the page pools, heads,
 * head_dim, page size and every policy stay the plan's). The new metadata
 * overwrites the workspace with one host-to-device copy on `stream`, which
 * the call waits for; a pod_run captured earlier on this handle and
 * workspace then computes the new plan when replayed (the caller updates the
 * tensors it captured, e.g. the cache pages and queries, in place).
 * Errors: POD_ERR_INVALID_ARG (no capacity mode, a table that fails pod_plan's
 * checks or exceeds a capacity), POD_ERR_WORKSPACE (no bound workspace),
 * POD_ERR_CUDA.
 */
pod_status pod_replan(pod_handle h, const int32_t* p_q_indptr, const int32_t* p_kv_indptr,
                      const int32_t* p_kv_indices, const int32_t* p_last_page_len,
                      int32_t p_batch, const int32_t* d_q_indptr, const int32_t* d_kv_indptr,
                      const int32_t* d_kv_indices, const int32_t* d_last_page_len,
                      int32_t d_batch, void* stream);

/* Release the handle (host memory only). NULL is accepted. Library
 * mechanics; no passage. */
pod_status pod_destroy(pod_handle h);

/* Thread-local message of the last error ("" if none). Valid until the next
 * call. Library mechanics; no passage. */
const char* pod_last_error(void);

/*
 * pod_read_device_status — synchronise `stream`, read and clear the device
 * status word in `workspace`. *device_status receives 0 when every kernel
 * finished its work; otherwise a bit mask (1 = a bounded wait of the prefill
 * pipeline ran out, 2 = shared-memory alignment check failed). Returns
 * POD_ERR_DEVICE_STATUS when the word was non-zero. Library mechanics (the
 * bounded waits report here instead of hanging); no passage.
 */
pod_status pod_read_device_status(pod_handle h, void* workspace, void* stream,
                                  int32_t* device_status);

/*
 * pod_plan_table — host copy of one plan table, for inspection and tests.
 * which: 0 = summary ints, 1 = prefill tiles, 2 = decode items, 3 = CTA work
 * offsets, 4 = CTA work list, 5 = merge groups, 6 = p kv_len, 7 = d kv_len,
 * 8 = prefill tile queue, 9 = decode item queue, 10 = decode queue records
 * (16 ints per queue position: the item record, then kv_len, first query row,
 * q_len, first page-table entry, page count of its request), 11 = first
 * custom-mask bit of each prefill request and the total, as int64 values
 * stored as little-endian int32 pairs (empty without a custom mask); under
 * RoPE, 12 / 13 = per page-table entry of the prefill / decode half the
 * position of its slot 0 and its slots below kv_len (2 ints; the decode half
 * has no page copies, so 13 is empty), 14 / 15 = the position of each
 * prefill / decode query row (empty without RoPE).
 * Copies min(count, capacity) int32 values into `out` (may be NULL to query
 * *count). Each table's record format is documented beside the planner
 * (csrc/pod_plan.h in the library sources). Library mechanics (plan
 * introspection for tests and tools); no passage.
 */
pod_status pod_plan_table(pod_handle h, int32_t which, int32_t* out, int64_t capacity,
                          int64_t* count);

/*
 * pod_run_static_scratch — pod_run for callers that cannot allocate device
 * memory. The paper has no counterpart: this entry point is a deployment aid
 * of this library.
 *
 * Some callers cannot call cudaMalloc: plugins whose host application owns all
 * device memory through its own pool, processes held to a fixed device-memory
 * budget, and serving loops that cannot take the implicit synchronisation of
 * cudaMalloc/cudaFree. This call needs no workspace from them: the scratch the
 * kernels use (plan metadata, split partials, status word) is a fixed
 * 32 MiB array inside the library (pod_static_scratch_capacity()), which every
 * GPU that loads the library holds until the process exits. The caller still
 * passes the input and output tensors, with the same meaning as for pod_run.
 *
 * Each call uploads the plan's metadata into that array (clearing the status
 * word) with a host-to-device copy, waits for the stream to finish that copy
 * (so every call blocks the host until the work queued before it on the
 * stream is done), and then runs the same kernels as pod_run. Every call on a device
 * shares the one array, which keeps the last call's contents: calls that
 * overlap on the GPU (other streams, other threads) race and must be
 * serialised by the caller. The handle becomes bound to the array (a later
 * pod_run on it must pass that array's address or re-bind with
 * pod_bind_workspace). The first call on a device looks up the array's device
 * address with that device current. No device memory is allocated or freed.
 *
 * Errors: POD_ERR_WORKSPACE (with a message) when pod_workspace_size(h)
 * exceeds the array; otherwise those of pod_bind_workspace and pod_run.
 */
pod_status pod_run_static_scratch(pod_handle h, const void* q_p, const void* kv_p,
                                  const void* q_d, const void* kv_d, const float* sinks,
                                  void* out_p, float* lse_p, void* out_d, float* lse_d,
                                  void* stream);

/* Size in bytes of the static scratch array used by pod_run_static_scratch.
 * Library mechanics; no passage. */
size_t pod_static_scratch_capacity(void);

#ifdef __cplusplus
}
#endif

#endif /* POD_GB300_H */
