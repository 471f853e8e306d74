// pod_plan.h — plan records shared by the host planner and the CUDA kernels.
//
// The plan is the "auxiliary data structure built once and reused by every
// run" of the POD walkthrough ("plan/run 生命周期"). Every table is int32 and
// lives, on the device, in the integer part of the caller's workspace.
//
// Record formats (POD_REC = 8 int32 per record)
//   prefill tile  : req, kv_head, tok0, ntok, kv_lo, kv_hi, prow, 0
//                   rows of the tile = ntok tokens x G qo heads (token-major),
//                   keys [kv_lo, kv_hi) of request `req`; prow = first partial
//                   row when the tile writes a split partial, -1 when it writes
//                   the final output.
//   decode item   : req, kv_head, tok0, ntok, k0, k1, prow, 0
//                   keys [k0, k1) of one (request, kv head, token group).
//   merge group   : half (0 prefill, 1 decode), req, kv_head, tok0, ntok,
//                   prow0, nsplit, R   with R = ntok * G; split j, row r of the
//                   group is partial row prow0 + j * R + r.
//   cta_ptr[grid+1], cta_list[]: the planner's static assignment, CTA c taking
//                   cta_list[cta_ptr[c] .. cta_ptr[c+1]) (prefill tiles when
//                   c < n_prefill_ctas, decode items otherwise); it sizes the
//                   CTA split and is kept for inspection.
//   pqueue[n_tiles], dqueue[n_items]: the work queues the kernel serves, every
//                   tile / item in decreasing cost. CTAs c < n_prefill_ctas
//                   take prefill tiles first, the others decode items first;
//                   a CTA whose queue runs dry helps with the other one. The
//                   queue heads are three counters in the status block
//                   (status[8] tiles, status[9] items, status[10] CTAs done);
//                   the last CTA to finish resets them to zero.
//   dqrec[n_items][16]: the decode queue again, one self-contained record per
//                   position: the item's record (8 ints), then kv_len,
//                   q_base (first query row), q_len, page_base (kv_indptr of
//                   the request), npages, 0, 0, 0. A CTA that takes queue
//                   position i reads only this record, so claiming an item
//                   costs one dependent load.
//   mrow_ptr[n_groups+1]: prefix sums of R over merge groups.
//   summary (pod_plan_table which = 0): see PodSummary below.
#pragma once
#include <cuda.h>
#include <stdint.h>
#include <vector_types.h>

// Status block: int32 words at the start of the workspace. [0] device status
// word; [8], [9], [10] the tile and item queue heads and the count of
// finished CTAs (the last CTA rewinds them); [16..20] the plan's counts
// below. In CUDA-graph capacity mode the merge kernel reads its counts here
// rather than from its launch parameters, so a launch captured once serves
// every later plan written into the same capacity-sized workspace.
#define POD_ST_NTILES 16   // prefill tiles in the queue
#define POD_ST_NITEMS 17   // decode items in the queue
#define POD_ST_NPCTAS 18   // CTAs that start on the prefill queue
#define POD_ST_NGROUPS 19  // merge groups
#define POD_ST_NMROWS 20   // merge rows

#define POD_REC 8
#define POD_DQREC 16
#define POD_TILE_ROWS 128      // prefill tile rows (tcgen05 M)
#define POD_KBLOCK 64          // keys per prefill KV block
#define POD_DECODE_ROWS 32     // max rows of a decode item (2 mma.sync m16 tiles)
#define POD_DECODE_STAGE 64    // keys per decode pipeline stage
#define POD_CTAS_PER_SM 2
// logits transform applied by both halves before masking and softmax
#define POD_LT_NONE 0
#define POD_LT_SOFTCAP 1   // cap * tanh(x / cap) of the scaled logit x
#define POD_LT_ALIBI 2     // + slope[head] * (t - p)

enum PodSummary {
  S_H = 0, S_HK, S_D, S_PS, S_CAUSAL, S_WINDOW, S_DTYPE, S_SINKS, S_NUM_SMS, S_GRID,
  S_NP_CTAS, S_ND_CTAS, S_NTILES, S_NITEMS, S_NGROUPS, S_NMROWS, S_NPROWS,
  S_P_ROWS, S_D_ROWS, S_P_BATCH, S_D_BATCH, S_DECODE_CHUNK, S_WS_LO, S_WS_HI,
  S_P_TMA, S_D_TMA, S_P_MASK, S_ROPE, S_COUNT
};

// Everything a kernel needs, passed by value at launch (as a __grid_constant__
// parameter, so that the tensor maps can be addressed by TMA instructions).
struct PodParams {
  // TMA descriptors: Q as [rows, H, d] (box 64 x G x tokens), the paged cache
  // as [pages, 2, ps, Hk, d] (box 64 x 1 x rows x 1 x pages); valid when the
  // half's *_tma flag is set (Q maps whenever the half is non-empty).
  CUtensorMap tm_q_p, tm_kv_p, tm_q_d, tm_kv_d;
  // RoPE: the low parts of the rotated queries, [rows, H, d] like tm_q_*
  CUtensorMap tm_qlo_p, tm_qlo_d;
  int p_tma, d_tma;          // keys per TMA K/V box of the half; 0 = cp.async gather
  int p_num_pages, d_num_pages;
  int tq, tu;                // tokens per prefill tile / per decode unit
  int H, Hk, G, d, ps, ps_shift, causal, window_left, has_sinks;
  // page layout of each half's cache: 0 = NHD pages [2, ps, Hk, d],
  // 1 = HND pages [2, Hk, ps, d] (only the cp.async gathers read it; the
  // tensor maps carry the layout in their strides)
  int p_hnd, d_hnd;
  // logits transform: lt = POD_LT_*; lt_c = cap / sm_scale (soft cap in raw
  // q.k units); lt_inv_scale = 1 / sm_scale; alibi = device [H] slopes
  int lt;
  float lt_c, lt_inv_scale;
  const float* alibi;
  float scale_log2;          // sm_scale * log2(e)
  // decode cache in FP8 E4M3 (head_dim 128): d_scale_log2 = scale_log2 * k_scale,
  // outputs multiplied by v_scale
  int d_fp8;
  float d_scale_log2, v_scale;
  int n_p_ctas, grid;
  int n_groups, n_mrows;
  int p_batch, d_batch;
  const int32_t *p_q_indptr, *p_kv_indptr, *p_kv_indices, *p_kv_len;
  const int32_t *d_q_indptr, *d_kv_indptr, *d_kv_indices, *d_kv_len;
  const int32_t *ptiles, *ditems, *cta_ptr, *cta_list, *mgroups, *mrow_ptr;
  const int32_t *pqueue, *dqueue, *dqrec;
  int n_tiles, n_items;
  // CUDA-graph capacity mode (1): n_tiles / n_items are the capacities (the
  // queues hold sentinels past the plan's own records), the merge kernel
  // takes its counts from the workspace status block and its grid covers
  // mrows_grid rows. A load of the counts per claim in the fused kernel
  // measured 1.6 % slower, so K1 takes them from these parameters.
  int counts_in_ws;
  int mrows_grid;
  float* part_o;             // [n_prows, d]
  float* part_lse;           // [n_prows]
  int32_t* status;           // device status word
  const void *q_p, *kv_p, *q_d, *kv_d;
  const float* sinks;
  // RoPE (ROPE_LLAMA): rope = 1; q_* point at the rotated high parts and
  // q_d_lo at the decode low parts; kv_p at the prefill copies (K_hi, V, K_lo
  // per page); rope_tab = (cos, sin) [rope_rows][d/2] of position x frequency
  int rope, rope_rows;
  const void* q_d_lo;
  const float2* rope_tab;
  // custom prefill mask (NULL = none): packed bits, little bit order, of each
  // request's [q_len, kv_len] matrix; p_mask_off[r] = request r's first bit
  const uint8_t* p_mask;
  const long long* p_mask_off;
  long long p_mask_bytes;
  void *out_p, *out_d;
  float *lse_p, *lse_d;
};
