// pod_kernels.cuh — the fused POD kernel for sm_103a (K1), as templates.
//
// Each variant family is instantiated in its own translation unit
// (pod_k1_plain.cu, pod_k1_lt.cu, pod_k1_rope.cu) so that they compile in
// parallel; pod_launch.cu holds the split merge (K2) and the dispatch.
//
// K1 `pod_kernel`: one persistent grid; CTA c < n_prefill_ctas runs prefill
// tiles, the other CTAs run decode items (POD walkthrough, "POD 是什么": one
// launch serves the compute-bound prefill and the memory-bound decode, so the
// two share the SMs instead of leaving gaps between two launches).
//
//  prefill tile (128 query rows = ntok tokens x G qo heads of one KV head):
//    warps 5-6  TMA producers (one thread each): the Q tile, then 64-key K
//               blocks (3-stage ring) and V blocks (2-stage ring) as page
//               boxes through the page table, 128B-swizzled by the hardware
//               (warps 5-7 gather with cp.async when the page table does not
//               allow page boxes);
//    warp 4     one thread issues tcgen05.mma: S = Q K^T into TMEM (double
//               buffered), then O += P V with P read from TMEM;
//    warps 0-3  one TMEM lane (= one query row) per thread: tcgen05.ld of S,
//               bottom-right causal / window mask, online softmax in base 2
//               with lazy rescaling of O, P packed to 16 bits and stored over
//               the S columns it came from, final O / (l + sink) and LSE.
//  decode item (<= 32 rows = q tokens x G heads, keys [k0, k1) of one chunk):
//    a 3-stage ring of 64-key K/V stages fed by TMA page boxes (or cp.async);
//    warp w owns m-tile w/4 and keys 16*(w%4).. of each stage and runs
//    mma.sync m16n8k16 for Q K^T and P V with an online softmax in registers;
//    warps combine through shared memory and write the final output, or an
//    fp32 partial (o, lse) when the plan split the KV range.
//
// ROPE_LLAMA (template flag RP, FlashInfer guide, "快速上手": pos_encoding_mode
// with rope_scale and rope_theta): queries arrive rotated, as a 16-bit high
// part and a 16-bit low part (q = q_hi + q_lo to about 16 bits of mantissa),
// from a pre-pass. The prefill keys arrive the same way (copies of the
// prefill pages, K_hi / V / K_lo per page). The decode keys are rotated in
// registers from the caller's cache, right after ldmatrix, in fp32, then
// split into high and low parts. Both halves form each logit from three
// products q_hi.k_hi + q_hi.k_lo + q_lo.k_hi, so no rotated operand is
// rounded to 16 bits. The RoPE kernel runs one CTA per SM: the low parts
// need the shared memory of a second CTA.
#pragma once
#include <cuda_runtime.h>
#include <math.h>

#include <atomic>
#include <mutex>

#include "pod_device.cuh"
#include "pod_launch.h"
#include "pod_plan.h"

using namespace pod;

namespace {

constexpr int kThreads = 256;

// ------------------------------------------------------------------ layouts
template <int D, bool RP>
struct PLayout {                                   // prefill shared memory
  static constexpr int NKB = D / 64;               // 64-element K blocks of head_dim
  static constexpr int QBLK = POD_TILE_ROWS * 128; // 128 rows x 128 B
  static constexpr int KVBLK = POD_KBLOCK * 128;   // 64 rows x 128 B
  static constexpr int KSTAGE = NKB * KVBLK;       // one 64-key K or V block
  static constexpr int NQ = RP ? 2 : 1;            // Q tile (RoPE: high, then low part)
  static constexpr int KSTEP = NQ * KSTAGE;        // K stage (RoPE: high, then low part)
  static constexpr int NK = 3, NV = 2;             // K and V stage rings
  static constexpr int Q_OFF = 0;
  static constexpr int QLO_OFF = Q_OFF + NKB * QBLK;
  static constexpr int K_OFF = Q_OFF + NQ * NKB * QBLK;
  static constexpr int V_OFF = K_OFF + NK * KSTEP;
  static constexpr int BAR_OFF = V_OFF + NV * KSTAGE;
  // BAR_OFF + 0: mbarriers, +224: TMEM address, +228: abort flag,
  // +256: tile-id ring [8], +288: published count, +320: per-warp read counts [8]
  static constexpr int TQ_OFF = BAR_OFF + 256;
  static constexpr int TOTAL = BAR_OFF + 384;
  // TMEM: S/P[2] (2 x 64 columns) then O (D columns); 256 columns let two
  // CTAs share an SM's 512, head_dim 256 takes them all (one CTA per SM)
  static constexpr int TM_S = 0, TM_O = 128;
  static constexpr int TMEM_COLS = TM_O + D <= 256 ? 256 : 512;
};

// CTAs per SM of an instantiation: RoPE (low parts of the rotated operands)
// and head_dim 256 (shared memory and TMEM) run one, the others two.
template <int D, bool RP>
constexpr int ctas_per_sm() {
  return (RP || D > 128) ? 1 : POD_CTAS_PER_SM;
}

template <int D, bool RP>
struct DLayout {                                   // decode shared memory
  static constexpr int NKB = D / 64;
  static constexpr int QDH = POD_DECODE_ROWS * 128; // one 64-column half of Q: 32 rows x 128 B
  static constexpr int KDH = POD_DECODE_STAGE * 128;// one half of a 64-key K or V block
  static constexpr int KBYTES = NKB * KDH;
  static constexpr int STAGE_BYTES = 2 * KBYTES;    // K then V
  // RoPE runs one CTA per SM: a deeper ring keeps the bytes in flight per SM
  static constexpr int NSTAGE = RP ? 6 : 3;
  static constexpr int NQ = RP ? 2 : 1;             // Q (RoPE: high, then low part)
  static constexpr int Q_OFF = 0;
  static constexpr int QLO_OFF = NKB * QDH;
  static constexpr int STAGE_OFF = NQ * NKB * QDH;
  static constexpr int BAR_OFF = STAGE_OFF + NSTAGE * STAGE_BYTES;
  // FP8 (E4M3) cache, head_dim 128 only: stages of 128 keys, [key][128 B]
  // codes per K or V (32 KB a stage, as a 16-bit stage), fed to e4m3 MMAs as
  // they are. Each item's Q is rewritten as up to three e4m3 parts of 32 rows
  // x 128 B: parts 0 and 1 over the 16-bit Q, part 2 after the barriers, then
  // one fp32 row scale per row.
  static constexpr bool F8OK = D == 128 && !RP;
  static constexpr int F8_KEYS = 2 * POD_DECODE_STAGE;
  static constexpr int F8_HALF = F8_KEYS * 128;            // K or V of a stage
  static constexpr int F8_STAGE = 2 * F8_HALF;
  static constexpr int Q8_PART = POD_DECODE_ROWS * 128;
  static constexpr int Q8X_OFF = BAR_OFF + 128;
  static constexpr int QSC_OFF = Q8X_OFF + Q8_PART;
  static constexpr int TOTAL = BAR_OFF + 128;                  // 16-bit cache
  static constexpr int TOTAL_F8 = QSC_OFF + POD_DECODE_ROWS * 16;  // FP8 cache
  static_assert(!F8OK || (F8_STAGE <= STAGE_BYTES && 2 * Q8_PART <= NKB * QDH),
                "FP8 stages and Q parts must fit the 16-bit ones");
  // combine scratch (reuses the stages): 8 warps x 16 rows x D floats, then m/l
  static constexpr int SCR_O = STAGE_OFF;
  static constexpr int SCR_ML = STAGE_OFF + 8 * 16 * D * 4;
  static_assert(SCR_ML + 8 * 16 * 2 * 4 <= BAR_OFF, "combine scratch must fit in the stages");
  static_assert(STAGE_OFF % 1024 == 0, "stages must be 1024-byte aligned");
  static_assert(NSTAGE * 8 <= 64, "stage barriers overlap the abort flag");
};

// Dynamic shared memory of an instantiation: the FP8 regions are requested
// only by the FP8 kernels (a larger request leaves less of the SM's L1).
template <int D, bool RP, bool F8 = false>
constexpr int smem_bytes() {
  constexpr int DT = F8 ? DLayout<D, RP>::TOTAL_F8 : DLayout<D, RP>::TOTAL;
  return PLayout<D, RP>::TOTAL > DT ? PLayout<D, RP>::TOTAL : DT;
}

POD_DEV void raise_status(int32_t* status, int code) { atomicOr(status, code); }

// All 32 lanes wait; the result is warp-uniform so that warp-collective
// tcgen05.ld / __any_sync calls after it are reached by every lane.
POD_DEV bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  const bool ok = mbar_wait(bar, parity, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// ============================================================ prefill role
// Barrier slots (8 bytes each) at PLayout::BAR_OFF.
enum {
  B_QFULL = 0, B_QEMPTY = 1,
  B_KFULL = 2,                     // [NK]
  B_KEMPTY = B_KFULL + 3,          // [NK]
  B_VFULL = B_KEMPTY + 3,          // [NV]
  B_VEMPTY = B_VFULL + 2,          // [NV]
  B_SFULL = B_VEMPTY + 2,          // [2] S_j of buffer j%2 computed
  B_PFULL = B_SFULL + 2,           // [2] P_j of buffer j%2 written into TMEM
  B_PVDONE = B_PFULL + 2,          // [2] PV_j (A = P_j) finished
  B_FINAL = B_PVDONE + 2,
  B_COUNT = B_FINAL + 1
};

// Runs prefill tiles from the shared queue until it is empty. Warp 5 takes
// tiles from the global queue and publishes them in order on a small ring in
// shared memory; every other warp that walks tiles reads the same sequence.
// Returns false when a wait ran out (the status word then says so).
template <typename T, int D, int LT, bool RP>
__device__ bool prefill_role(const PodParams& P, uint8_t* smem, uint32_t tmem) {
  using L = PLayout<D, RP>;
  constexpr int NK = L::NK, NV = L::NV;
  static_assert(NK == 3 && NV == 2, "the barrier slots below are laid out for 3 K and 2 V stages");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + L::BAR_OFF;
  auto BAR = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::BAR_OFF + 228);
  static_assert(B_COUNT * 8 <= 224, "barriers overlap the TMEM slot");
  volatile int* tq_ring = reinterpret_cast<volatile int*>(smem + L::TQ_OFF);
  volatile int* tq_pub = tq_ring + 8;
  volatile int* tq_used = tq_ring + 16;
  constexpr int kNever = 1 << 30;

  // warp 5: take the next tile of the global queue and publish it as number seq
  // (-1: queue empty, -2: gave up waiting for a reader)
  auto fetch_tile = [&](int seq) -> int {
    int id = -1;
    if (lane == 0) {
      // (in CUDA-graph capacity mode n_tiles is the capacity and the queue
      // holds -1 past the plan's own tiles: the queue is empty there too)
      const int idx = atomicAdd(P.status + 8, 1);
      id = idx < P.n_tiles ? __ldg(P.pqueue + idx) : -1;
      const uint64_t t0 = globaltimer();
      for (int r = 0; r < 8 && id != -2; ++r)
        while (tq_used[r] < seq - 7)
          if (*abort_flag || globaltimer() - t0 > POD_WAIT_TIMEOUT_NS) { id = -2; break; }
      if (id != -2) {
        tq_ring[seq & 7] = id;
        __threadfence_block();
        *tq_pub = seq + 1;
      }
    }
    return __shfl_sync(0xffffffffu, id, 0);
  };
  // any other warp: the tile published as number seq (lane 0 reads, the warp shares)
  auto read_tile = [&](int seq, bool lone_lane) -> int {
    int id = -1;
    if (lane == 0) {
      const uint64_t t0 = globaltimer();
      while (*tq_pub <= seq)
        if (*abort_flag || globaltimer() - t0 > POD_WAIT_TIMEOUT_NS) { id = -2; break; }
      if (id != -2) {
        __threadfence_block();
        id = tq_ring[seq & 7];
        tq_used[warp] = seq + 1;
      }
    }
    return lone_lane ? id : __shfl_sync(0xffffffffu, id, 0);
  };

  if (tid == 0) {
    const uint32_t kv_arrivals = P.p_tma ? 1u : 96u;  // TMA: one expect_tx arrive
    mbar_init(BAR(B_QFULL), 1);
    mbar_init(BAR(B_QEMPTY), 1);
    for (int s = 0; s < NK; ++s) {
      mbar_init(BAR(B_KFULL + s), kv_arrivals);
      mbar_init(BAR(B_KEMPTY + s), 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(BAR(B_VFULL + s), kv_arrivals);
      mbar_init(BAR(B_VEMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(BAR(B_SFULL + b), 1);
      mbar_init(BAR(B_PFULL + b), 128);
      mbar_init(BAR(B_PVDONE + b), 1);
    }
    mbar_init(BAR(B_FINAL), 1);
    *abort_flag = 0;
    *tq_pub = 0;
    for (int r = 0; r < 8; ++r) tq_used[r] = 0;
    tq_used[5] = kNever;                       // the fetcher itself
    if (P.p_tma) tq_used[7] = kNever;          // idle when TMA feeds the tiles
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int G = P.G, H = P.H;

  if (warp >= 5) {
    // ------------------------------------------------------------ loaders
    fence_proxy_async();  // generic accesses of an earlier decode phase come first
    int kfill = 0, vfill = 0, qfill = 0;
    // L2 priorities: a Q tile is read once; the prefill K/V blocks are re-read
    // by every tile of their request and head, next to a decode stream that
    // would otherwise evict them. (Each policy is made where it is used, one
    // instruction, rather than held in registers across the loops.)
#define pol_q l2_policy_evict_first()
#define pol_kv l2_policy_evict_last()
    bool ok = true;
    const uint32_t q_bytes = (uint32_t)(L::NQ * L::NKB * 128 * G * P.tq);
    if (P.p_tma) {
      // warp 5 fetches Q and K, warp 6 fetches V, each running ahead on its own
      // ring. Lane i looks up the page of box group i and issues its boxes, so
      // the page-table reads of one block overlap. Page ids beyond the request
      // map to an out-of-range page coordinate, which TMA fills with zeros.
      if (warp == 5 || warp == 6) {
        const bool is_v = warp == 6;
        const void* tkv = &P.tm_kv_p;
        if (lane == 0) tma_prefetch_desc(tkv);
        const int ngroups = POD_KBLOCK / P.p_tma;
        for (int seq = 0; ok; ++seq) {
          const int tile = is_v ? read_tile(seq, false) : fetch_tile(seq);
          if (tile == -2) { ok = false; break; }
          if (tile < 0) break;
          const int32_t* rec = P.ptiles + POD_REC * tile;
          const int req = rec[0], g = rec[1], tok0 = rec[2], lo = rec[4], hi = rec[5];
          const int page_base = P.p_kv_indptr[req];
          const int npages = P.p_kv_indptr[req + 1] - page_base;
          if (!is_v) {
            if (!warp_wait(BAR(B_QEMPTY), (qfill & 1) ^ 1, abort_flag)) { ok = false; break; }
            if (lane == 0) {
              mbar_arrive_expect_tx(BAR(B_QFULL), q_bytes);
              for (int dh = 0; dh < L::NKB; ++dh) {
                tma_load_3d_hint(sbase + L::Q_OFF + dh * L::QBLK, &P.tm_q_p, dh * 64, g * G,
                                 P.p_q_indptr[req] + tok0, BAR(B_QFULL), pol_q);
                if (RP)
                  tma_load_3d_hint(sbase + L::QLO_OFF + dh * L::QBLK, &P.tm_qlo_p, dh * 64, g * G,
                                   P.p_q_indptr[req] + tok0, BAR(B_QFULL), pol_q);
              }
            }
            ++qfill;
          }
          const int b0 = (lo / POD_KBLOCK) * POD_KBLOCK;
          const int nb = (hi - b0 + POD_KBLOCK - 1) / POD_KBLOCK;
          for (int j = 0; j < nb; ++j) {
            const int NS = is_v ? NV : NK;
            const int fill = is_v ? vfill : kfill;
            const int s = fill % NS;
            const int empty = (is_v ? B_VEMPTY : B_KEMPTY) + s, full = (is_v ? B_VFULL : B_KFULL) + s;
            if (!warp_wait(BAR(empty), ((fill / NS) & 1) ^ 1, abort_flag)) { ok = false; break; }
            if (lane == 0) mbar_arrive_expect_tx(BAR(full), (uint32_t)(is_v ? L::KSTAGE : L::KSTEP));
            __syncwarp();
            const uint32_t dst0 = is_v ? sbase + L::V_OFF + s * L::KSTAGE : sbase + L::K_OFF + s * L::KSTEP;
            const int kb = b0 + j * POD_KBLOCK;
            for (int gi = lane; gi < ngroups; gi += 32) {
              const int o = gi * P.p_tma;
              const int t = kb + o;
              const int pidx = t >> P.ps_shift;
              const int page = pidx < npages ? __ldg(P.p_kv_indices + page_base + pidx) : P.p_num_pages;
              const int tin = P.ps >= 8 ? (t & (P.ps - 1)) : 0;
              for (int dh = 0; dh < L::NKB; ++dh) {
                tma_load_5d_hint(dst0 + dh * L::KVBLK + o * 128, tkv, dh * 64, g, tin, is_v ? 1 : 0,
                                 page, BAR(full), pol_kv);
                // RoPE copies hold K_hi, V, K_lo per page: the low part is row 2
                if (RP && !is_v)
                  tma_load_5d_hint(dst0 + L::KSTAGE + dh * L::KVBLK + o * 128, tkv, dh * 64, g, tin, 2,
                                   page, BAR(full), pol_kv);
              }
            }
            if (is_v) ++vfill; else ++kfill;
          }
        }
      }
    } else {
      // cp.async gather by warps 5-7 (96 threads); Q still comes by TMA
      const int lt = tid - 160;  // 0..95
      const T* __restrict__ kvg = reinterpret_cast<const T*>(P.kv_p);
      const size_t vstride = (size_t)P.ps * P.Hk * D;   // K row -> V row of the same page
      constexpr int NKV = RP ? 3 : 2;                    // rows per page (RoPE: K_hi, V, K_lo)
      constexpr int KCH = POD_KBLOCK * (D / 8);
      constexpr int PER = (KCH + 95) / 96;
      for (int seq = 0; ok; ++seq) {
        const int tile = warp == 5 ? fetch_tile(seq) : read_tile(seq, false);
        if (tile == -2) { ok = false; break; }
        if (tile < 0) break;
        const int32_t* rec = P.ptiles + POD_REC * tile;
        const int req = rec[0], g = rec[1], tok0 = rec[2], lo = rec[4], hi = rec[5];
        const int page_base = P.p_kv_indptr[req];
        if (lt == 0) {
          if (!mbar_wait(BAR(B_QEMPTY), (qfill & 1) ^ 1, abort_flag)) ok = false;
          if (ok) {
            mbar_arrive_expect_tx(BAR(B_QFULL), q_bytes);
            for (int dh = 0; dh < L::NKB; ++dh) {
              tma_load_3d_hint(sbase + L::Q_OFF + dh * L::QBLK, &P.tm_q_p, dh * 64, g * G,
                               P.p_q_indptr[req] + tok0, BAR(B_QFULL), pol_q);
              if (RP)
                tma_load_3d_hint(sbase + L::QLO_OFF + dh * L::QBLK, &P.tm_qlo_p, dh * 64, g * G,
                                 P.p_q_indptr[req] + tok0, BAR(B_QFULL), pol_q);
            }
          }
        }
        ++qfill;
        if (!ok) break;
        const int b0 = (lo / POD_KBLOCK) * POD_KBLOCK;
        const int nb = (hi - b0 + POD_KBLOCK - 1) / POD_KBLOCK;
        // one K or V block: page ids first (independent loads), then the copies
        auto load_block = [&](int j, bool is_v, uint32_t dst_base) {
          const int kb = b0 + j * POD_KBLOCK;
          int pages[PER];
#pragma unroll
          for (int i = 0; i < PER; ++i) {
            const int idx = lt + 96 * i;
            const int key = (idx < KCH ? idx : 0) / (D / 8);
            const int t = kb + key;
            const int tt = t < hi ? t : kb;
            const int pg_i = P.ps_shift >= 0 ? (tt >> P.ps_shift) : (tt / P.ps);
            pages[i] = __ldg(P.p_kv_indices + page_base + pg_i);
          }
#pragma unroll
          for (int i = 0; i < PER; ++i) {
            const int idx = lt + 96 * i;
            if (idx < KCH) {
              const int key = idx / (D / 8), c = idx % (D / 8);
              const int t = kb + key;
              const bool valid = t < hi;
              const int tt = valid ? t : kb;
              const int slot = P.ps_shift >= 0 ? (tt & (P.ps - 1)) : (tt % P.ps);
              const T* src = kvg + (P.p_hnd
                  ? (((size_t)pages[i] * NKV * P.Hk + g) * P.ps + slot) * D + c * 8
                  : (((size_t)pages[i] * NKV * P.ps + slot) * P.Hk + g) * D + c * 8);
              cp_async16_hint(dst_base + (c >> 3) * L::KVBLK + sw128_off(key, c & 7),
                              is_v ? src + vstride : src, valid ? 16u : 0u, pol_kv);
              if (RP && !is_v)
                cp_async16_hint(dst_base + L::KSTAGE + (c >> 3) * L::KVBLK + sw128_off(key, c & 7),
                                src + 2 * vstride, valid ? 16u : 0u, pol_kv);
            }
          }
        };
        for (int st = 0; st <= nb && ok; ++st) {
          if (st < nb) {
            const int s = kfill % NK;
            if (!mbar_wait(BAR(B_KEMPTY + s), ((kfill / NK) & 1) ^ 1, abort_flag)) { ok = false; break; }
            load_block(st, false, sbase + L::K_OFF + s * L::KSTEP);
            cp_async_mbar_arrive(BAR(B_KFULL + s));
            ++kfill;
          }
          if (st > 0) {
            const int s = vfill % NV;
            if (!mbar_wait(BAR(B_VEMPTY + s), ((vfill / NV) & 1) ^ 1, abort_flag)) { ok = false; break; }
            load_block(st - 1, true, sbase + L::V_OFF + s * L::KSTAGE);
            cp_async_mbar_arrive(BAR(B_VFULL + s));
            ++vfill;
          }
        }
      }
      cp_async_wait_all();
    }
    if (!ok) {
      *abort_flag = 1;
      raise_status(P.status, POD_STATUS_TIMEOUT);
    }
#undef pol_q
#undef pol_kv
  } else if (warp == 4) {
    // ------------------------------------------------------------ MMA issuer
    // Order per tile: QK_0, [QK_1, PV_0], [QK_2, PV_1], ..., PV_{nb-1}. QK_{j+2}
    // reuses the TMEM columns of S_j / P_j; it is issued after PV_j by this one
    // thread, and MMAs issued by one thread run in order.
    if (lane == 0) {
      const bool bf16 = Pack<T>::kBF16;
      const uint32_t id_qk = idesc_f16(bf16, 128, POD_KBLOCK, false, false);
      const uint32_t id_pv = idesc_f16(bf16, 128, D, false, true);
      int kuse = 0, vuse = 0, qfill = 0, sc0 = 0;
      bool ok = true;
      for (int seq = 0; ok; ++seq) {
        const int tile = read_tile(seq, true);
        if (tile == -2) { ok = false; break; }
        if (tile < 0) break;
        const int32_t* rec = P.ptiles + POD_REC * tile;
        const int req = rec[0], lo = rec[4], hi = rec[5];
        const int kv_len = P.p_kv_len[req];
        const int b0 = (lo / POD_KBLOCK) * POD_KBLOCK;
        const int nb = (hi - b0 + POD_KBLOCK - 1) / POD_KBLOCK;
        if (!mbar_wait(BAR(B_QFULL), qfill & 1, abort_flag)) { ok = false; break; }
        ++qfill;
        for (int j = 0; j <= nb && ok; ++j) {
          if (j < nb) {
            const int s = kuse % NK;
            if (!mbar_wait(BAR(B_KFULL + s), (kuse / NK) & 1, abort_flag)) { ok = false; break; }
            tc_fence_after();
            // cp.async writes belong to the generic proxy: make them visible to
            // the MMA (async proxy). TMA writes need no fence.
            if (!P.p_tma) fence_proxy_async();
            const int b = (sc0 + j) & 1;
            const uint32_t qa = sbase + L::Q_OFF;
            const uint32_t ka = sbase + L::K_OFF + s * L::KSTEP;
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
              const uint32_t qo = (k >> 2) * L::QBLK + (k & 3) * 32;
              const uint32_t ko = (k >> 2) * L::KVBLK + (k & 3) * 32;
              const uint64_t ad = sdesc_sw128(qa + qo, 16, 1024);
              const uint64_t bd = sdesc_sw128(ka + ko, 16, 1024);
              mma_f16_ss(tmem + L::TM_S + b * POD_KBLOCK, ad, bd, id_qk, k > 0 ? 1u : 0u);
              if (RP) {
                // q.k = q_hi.k_hi + q_hi.k_lo + q_lo.k_hi (q_lo.k_lo is below fp32 rounding)
                const uint64_t adl = sdesc_sw128(qa + (L::QLO_OFF - L::Q_OFF) + qo, 16, 1024);
                const uint64_t bdl = sdesc_sw128(ka + L::KSTAGE + ko, 16, 1024);
                mma_f16_ss(tmem + L::TM_S + b * POD_KBLOCK, ad, bdl, id_qk, 1u);
                mma_f16_ss(tmem + L::TM_S + b * POD_KBLOCK, adl, bd, id_qk, 1u);
              }
            }
            mma_commit(BAR(B_SFULL + b));
            mma_commit(BAR(B_KEMPTY + s));
            if (j == nb - 1) mma_commit(BAR(B_QEMPTY));
            ++kuse;
          }
          if (j > 0) {
            // O += P_{j-1} V_{j-1}, P_{j-1} read from TMEM (columns of S_{j-1})
            const int i = j - 1;
            const int sc = sc0 + i;
            const int b = sc & 1;
            const int s = vuse % NV;
            if (!mbar_wait(BAR(B_VFULL + s), (vuse / NV) & 1, abort_flag)) { ok = false; break; }
            if (!mbar_wait(BAR(B_PFULL + b), (sc >> 1) & 1, abort_flag)) { ok = false; break; }
            tc_fence_after();
            const uint32_t va = sbase + L::V_OFF + s * L::KSTAGE;
            // 16-key steps past hi carry P = 0 for every row: skip them. Rows at
            // or past kv_len inside the last step come from unused slots of the
            // request's last page (TMA copies whole pages): zero them so that
            // P = 0 never meets a non-finite value.
            const int kb_i = b0 + i * POD_KBLOCK;
            const int ksteps = (min(hi, kb_i + POD_KBLOCK) - kb_i + 15) >> 4;
            const bool zero_tail = P.p_tma && kb_i + ksteps * 16 > kv_len;
            if (zero_tail) {
              for (int rr = kv_len - kb_i; rr < ksteps * 16; ++rr)
                for (int dh = 0; dh < L::NKB; ++dh)
                  for (int c = 0; c < 8; ++c)
                    asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(
                                     va + dh * L::KVBLK + sw128_off(rr, c)),
                                 "r"(0u)
                                 : "memory");
            }
            // generic writes (cp.async stage, zeroed tail) -> visible to the MMA
            if (!P.p_tma || zero_tail) fence_proxy_async();
            for (int k = 0; k < ksteps; ++k) {
              const uint64_t bd = sdesc_sw128(va + k * 2048, L::KVBLK, 1024);
              mma_f16_ts(tmem + L::TM_O, tmem + L::TM_S + b * POD_KBLOCK + k * 8, bd, id_pv,
                         (i > 0 || k > 0) ? 1u : 0u);
            }
            mma_commit(BAR(B_PVDONE + b));
            mma_commit(BAR(B_VEMPTY + s));
            ++vuse;
          }
        }
        sc0 += nb;
      }
      if (!ok) {
        *abort_flag = 1;
        raise_status(P.status, POD_STATUS_TIMEOUT);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int r = tid;  // query row of the tile == TMEM lane
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    T* __restrict__ outg = reinterpret_cast<T*>(P.out_p);
    int sc0 = 0;
    bool ok = true;
    const float NEG_INF = -INFINITY;
    for (int seq = 0; ok; ++seq) {
      const int tile = read_tile(seq, false);
      if (tile == -2) { ok = false; break; }
      if (tile < 0) break;
      const int32_t* rec = P.ptiles + POD_REC * tile;
      const int req = rec[0], g = rec[1], tok0 = rec[2], ntok = rec[3], lo = rec[4], hi = rec[5];
      const int prow = rec[6];
      const int kv_len = P.p_kv_len[req];
      const int q_len = P.p_q_indptr[req + 1] - P.p_q_indptr[req];
      const int nrows = ntok * G;
      const bool valid = r < nrows;
      const int tok = tok0 + (valid ? r / G : ntok - 1);
      const int head = g * G + (valid ? r % G : 0);
      const int pdiag = kv_len - q_len + tok;
      // a custom mask takes the place of the causal rule
      const bool masked = P.p_mask != nullptr;
      const int row_hi = (P.causal && !masked) ? min(pdiag + 1, kv_len) : kv_len;
      const int row_lo = P.window_left >= 0 ? max(pdiag - P.window_left, 0) : 0;
      const long long mrow = masked ? P.p_mask_off[req] + (long long)tok * kv_len : 0;
      // ALiBi: slope of this row's head in raw q.k units
      float a_slope = 0.f;
      if constexpr (LT == POD_LT_ALIBI) a_slope = __ldg(P.alibi + head) * P.lt_inv_scale;
      const int b0 = (lo / POD_KBLOCK) * POD_KBLOCK;
      const int nb = (hi - b0 + POD_KBLOCK - 1) / POD_KBLOCK;
      float m_ref = NEG_INF, l = 0.f;
      for (int j = 0; j < nb; ++j) {
        const int kb = b0 + j * POD_KBLOCK;
        const int sc = sc0 + j;
        const int b = sc & 1;
        if (!warp_wait(BAR(B_SFULL + b), (sc >> 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t s_addr = tmem + lane_base + L::TM_S + b * POD_KBLOCK;
        float s[POD_KBLOCK];
        tmem_ld64(s_addr, s);
        // (the RoPE kernel takes the soft cap as a run-time switch)
        if (LT == POD_LT_SOFTCAP || (RP && P.lt == POD_LT_SOFTCAP)) {
          // cap * tanh(x / cap) of the scaled logit, kept in raw q.k units
          const float c = P.lt_c, ic = 1.f / P.lt_c;
#pragma unroll
          for (int i = 0; i < POD_KBLOCK; ++i) s[i] = soft_cap(s[i], c, ic);
        }
        if constexpr (LT == POD_LT_ALIBI) {
          const float base = (float)(kb - pdiag);
#pragma unroll
          for (int i = 0; i < POD_KBLOCK; ++i) s[i] = fmaf(a_slope, base + (float)i, s[i]);
        }
        const bool full = (kb >= row_lo) && (kb + POD_KBLOCK <= row_hi);
        if (!full) {
#pragma unroll
          for (int i = 0; i < POD_KBLOCK; ++i) {
            const int t = kb + i;
            if (t < row_lo || t >= row_hi) s[i] = NEG_INF;
          }
        }
        if (masked) {
          // keys past kv_len read the next row's bits; row_hi has masked them
          const uint64_t bits = load_bits64(P.p_mask, P.p_mask_bytes, mrow + kb);
#pragma unroll
          for (int i = 0; i < POD_KBLOCK; ++i)
            if (!((bits >> i) & 1ull)) s[i] = NEG_INF;
        }
        // row max with three-input max: four independent chains over s[4..59]
        // (seven steps of eight), then s[60..63] one per chain
        static_assert(POD_KBLOCK == 64, "the max chains cover 64 columns");
        float c0 = s[0], c1 = s[1], c2 = s[2], c3 = s[3];
#pragma unroll
        for (int i = 4; i + 8 <= POD_KBLOCK; i += 8) {
          c0 = max3(c0, s[i], s[i + 1]);
          c1 = max3(c1, s[i + 2], s[i + 3]);
          c2 = max3(c2, s[i + 4], s[i + 5]);
          c3 = max3(c3, s[i + 6], s[i + 7]);
        }
        const float bmax = max3(max3(c0, c1, s[60]), max3(c2, c3, s[61]), fmaxf(s[62], s[63]));
        const float scale = P.scale_log2;
        const float m_new = fmaxf(m_ref, bmax * scale);
        const bool rescale = m_new > m_ref + 8.0f;   // also true for the first finite max
        const float m_use = rescale ? m_new : m_ref;
        const float m_sub = (m_use == NEG_INF) ? 0.f : m_use;
        float rs = 0.f;
        uint32_t pk[POD_KBLOCK / 2];
#pragma unroll
        for (int i = 0; i < POD_KBLOCK; i += 2) {
          const float e0 = ex2(fmaf(s[i], scale, -m_sub)), e1 = ex2(fmaf(s[i + 1], scale, -m_sub));
          rs += e0 + e1;
          pk[i / 2] = Pack<T>::two(e0, e1);
        }
        const bool need = rescale && (m_ref != NEG_INF) && j > 0;
        if (__any_sync(0xffffffffu, need)) {
          // O holds PV up to block j-1: wait for PV_{j-1}, then rescale it in TMEM
          const int sp = sc - 1;
          if (!warp_wait(BAR(B_PVDONE + (sp & 1)), (sp >> 1) & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const float alpha = need ? ex2(m_ref - m_use) : 1.f;
#pragma unroll 1
          for (int c = 0; c < D; c += 32) {
            float o[32];
            tmem_ld32(tmem + lane_base + L::TM_O + c, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tmem_st32(tmem + lane_base + L::TM_O + c, o);
          }
          l *= alpha;
        }
        m_ref = m_use;
        l += rs;
        // P_j (packed 16-bit pairs) over the first 32 columns of S_j: A operand of PV_j
        tmem_st32u(s_addr, pk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(BAR(B_PFULL + b));
      }
      if (!ok) break;
      {
        const int sl = sc0 + nb - 1;
        if (!warp_wait(BAR(B_PVDONE + (sl & 1)), (sl >> 1) & 1, abort_flag)) { ok = false; break; }
      }
      tc_fence_after();
      sc0 += nb;
      // epilogue: every lane loads (tcgen05.ld is warp-collective), valid rows store
      float denom = l;
      if (P.has_sinks && prow < 0) denom += ex2(P.sinks[head] * 1.4426950408889634f - m_ref);
      const float inv = (denom > 0.f) ? 1.f / denom : 0.f;
      const size_t orow = (size_t)(P.p_q_indptr[req] + tok) * H + head;
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        float o[32];
        tmem_ld32(tmem + lane_base + L::TM_O + c, o);
        if (valid) {
          if (prow < 0) {
            T* dst = outg + orow * D + c;
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
              uint4 v;
              v.x = Pack<T>::two(o[i + 0] * inv, o[i + 1] * inv);
              v.y = Pack<T>::two(o[i + 2] * inv, o[i + 3] * inv);
              v.z = Pack<T>::two(o[i + 4] * inv, o[i + 5] * inv);
              v.w = Pack<T>::two(o[i + 6] * inv, o[i + 7] * inv);
              *reinterpret_cast<uint4*>(dst + i) = v;
            }
          } else {
            float* dst = P.part_o + (size_t)(prow + r) * D + c;
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              *reinterpret_cast<float4*>(dst + i) =
                  make_float4(o[i] * inv, o[i + 1] * inv, o[i + 2] * inv, o[i + 3] * inv);
          }
        }
      }
      if (valid) {
        const float lse = (l > 0.f) ? m_ref + log2f(l) : NEG_INF;
        if (prow < 0) {
          if (P.lse_p) P.lse_p[orow] = lse;
        } else {
          P.part_lse[prow + r] = lse;
        }
      }
      tc_fence_before();
    }
    if (!ok) {
      *abort_flag = 1;
      raise_status(P.status, POD_STATUS_TIMEOUT);
    }
  }

  // ------------------------------------------------------------ teardown
  // every MMA of this role has finished before the CTA moves on (TMEM and the
  // shared memory may be reused)
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    if (lane == 0) mma_commit(BAR(B_FINAL));
    __syncwarp();
    int never = 0;  // wait for the MMAs even after an abort, still bounded by the timeout
    mbar_wait(BAR(B_FINAL), 0, (volatile int*)&never);
    tc_fence_after();
  }
  __syncthreads();
  const bool clean = *abort_flag == 0;
  if (tid == 0 && clean)
    for (int i = 0; i < B_COUNT; ++i) mbar_inval(BAR(i));
  return clean;
}

// ============================================================ decode role
// decode_role (16-bit caches) and decode_role_f8 (FP8 caches) run decode
// items from the shared queue until it is empty. They return false when a
// wait ran out (the status word then says so).
//
// One FP8 decode stage of one warp: 16 rows (m-tile mt) x KSL = 32 keys
// (slice ks of a 128-key stage), both products on e4m3 tensor cores.
// K and V stay the cache's codes. Q enters as NP e4m3 parts of the row scaled
// by 2^e (qp0 + p * qpart for parts 0-1, qp2 for part 2) and every logit sums
// the parts' products, fp32 accumulate. The row info at `rowinfo` (16 bytes
// a row: key range [lo, hi), then the softmax scale with 2^-e folded in)
// masks and scales rows g and g + 8. P is carried as 256 P (largest 256 <= 448) and
// split into an E4M3 high part and an E4M3 remainder, both multiplied into O.
// Key order inside an MMA: the accumulator gives a thread keys 8n + 2t +
// {0, 1} (n-tile n); its A words use slots 4t..4t+3 for keys {2t, 2t+1, 8+2t,
// 9+2t} and slots 16+4t.. for {16+2t, 17+2t, 24+2t, 25+2t}, and the V words
// are byte-permuted from ldmatrix.trans tiles into the same order.
template <bool BF16, int D, int KSL>
__device__ __forceinline__ void decode_stage_f8(uint32_t sk, int vhalf, uint32_t qp0, int qpart,
                                                uint32_t qp2, int mt, int ks, int lane, int kbase,
                                                int kv_len, uint32_t rowinfo,
                                                float (&m)[2], float (&l)[2], float (&o)[D / 8][4]) {
  int row_lo[2], row_hi[2];
  float sc[2];
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    const uint32_t a = rowinfo + (uint32_t)(mt * 16 + (lane >> 2) + 8 * h2) * 16u;
    asm volatile("ld.shared.v2.s32 {%0, %1}, [%2];" : "=r"(row_lo[h2]), "=r"(row_hi[h2]) : "r"(a));
    asm volatile("ld.shared.f32 %0, [%1 + 8];" : "=f"(sc[h2]) : "r"(a));
  }
  static_assert(KSL == 32 && D == 128, "FP8 stages are 32 keys per warp at head_dim 128");
  constexpr int NP = BF16 ? 2 : 3;
  const float NEG_INF = -INFINITY;
  float s[4][4];
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
  // ---- S = Q K^T: per 32-d step, two ldmatrix.x4 give the B words of the 4
  // n-tiles (keys 16 np + 8 (lane/16) + lane%8, 16-byte chunk 2j + (lane/8)%2)
#pragma unroll
  for (int j = 0; j < D / 32; ++j) {
    uint32_t kf[2][4];
#pragma unroll
    for (int np = 0; np < 2; ++np) {
      const int key = ks * KSL + np * 16 + (lane & 7) + ((lane >> 4) << 3);
      const int ch = 2 * j + ((lane >> 3) & 1);
      ldsm_x4(sk + key * 128 + ((ch ^ (key & 7)) << 4), kf[np][0], kf[np][1], kf[np][2], kf[np][3]);
    }
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      const int rr = mt * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
      const int ch = 2 * j + (lane >> 4);
      const uint32_t qb = p < 2 ? qp0 + p * qpart : qp2;
      uint32_t a[4];
      ldsm_x4(qb + rr * 128 + ((ch ^ (rr & 7)) << 4), a[0], a[1], a[2], a[3]);
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
        mma16832_e4m3(s[nt], a, kf[nt >> 1][2 * (nt & 1)], kf[nt >> 1][2 * (nt & 1) + 1]);
    }
  }
  // ---- mask (only where some key of the slice is outside a row's range),
  // online softmax in base 2
  const int kq = kbase + 2 * (lane & 3);
  const bool inner = __all_sync(0xffffffffu, kbase >= row_lo[0] && kbase >= row_lo[1] &&
                                                 kbase + KSL <= row_hi[0] && kbase + KSL <= row_hi[1]);
  float alpha[2];
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    float mm = NEG_INF;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float x = s[nt][2 * h2 + e];
        if (!inner) {
          const int key = kq + 8 * nt + e;
          if (key < row_lo[h2] || key >= row_hi[h2]) x = NEG_INF;
          s[nt][2 * h2 + e] = x;
        }
        mm = fmaxf(mm, x);
      }
    mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, 1));
    mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, 2));
    const float m_new = fmaxf(m[h2], mm * sc[h2]);
    const float m_sub = (m_new == NEG_INF) ? 0.f : m_new;
    alpha[h2] = ex2(m[h2] - m_sub);
    m[h2] = m_new;
    const float off = 8.f - m_sub;  // 256 P
    float sum = 0.f;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float pv = ex2(fmaf(s[nt][2 * h2 + e], sc[h2], off));
        s[nt][2 * h2 + e] = pv;
        sum += pv;
      }
    l[h2] = l[h2] * alpha[h2] + sum;
  }
  // a running max that did not move leaves alpha = 1 on every row of the warp
  if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      o[i][0] *= alpha[0];
      o[i][1] *= alpha[0];
      o[i][2] *= alpha[1];
      o[i][3] *= alpha[1];
    }
  }
  // ---- A words of 256 P: rows g (words 0, 2) and g + 8 (1, 3)
  uint32_t ph[4], pl[4];
  e4m3_hi_lo4(s[0][0], s[0][1], s[1][0], s[1][1], ph[0], pl[0]);
  e4m3_hi_lo4(s[0][2], s[0][3], s[1][2], s[1][3], ph[1], pl[1]);
  e4m3_hi_lo4(s[2][0], s[2][1], s[3][0], s[3][1], ph[2], pl[2]);
  e4m3_hi_lo4(s[2][2], s[2][3], s[3][2], s[3][3], ph[3], pl[3]);
  // ---- O += P V over the 8 16-byte d chunks. ldmatrix.trans of keys 8i..8i+7
  // (i = lane/8) gives a thread bytes (key 8i+2t, 8i+2t+1) x (d 2g, 2g+1);
  // the even-d and odd-d bytes make two n8 tiles: o[2c] holds d 16c + 4t +
  // {0, 2}, o[2c+1] d 16c + 4t + {1, 3}. Keys at or past kv_len may be unused
  // slots of the last page: their V bytes are zeroed so that P = 0 never
  // meets a NaN code.
  auto pv = [&](uint32_t vm0, uint32_t vm1) {
#pragma unroll
    for (int c = 0; c < D / 16; ++c) {
      const int key = ks * KSL + lane;
      uint32_t r0, r1, r2, r3;
      ldsm_x4_t(sk + vhalf + key * 128 + ((c ^ (key & 7)) << 4), r0, r1, r2, r3);
      const uint32_t be0 = __byte_perm(r0, r1, 0x6420) & vm0, be1 = __byte_perm(r2, r3, 0x6420) & vm1;
      const uint32_t bo0 = __byte_perm(r0, r1, 0x7531) & vm0, bo1 = __byte_perm(r2, r3, 0x7531) & vm1;
      mma16832_e4m3(o[2 * c], ph, be0, be1);
      mma16832_e4m3(o[2 * c], pl, be0, be1);
      mma16832_e4m3(o[2 * c + 1], ph, bo0, bo1);
      mma16832_e4m3(o[2 * c + 1], pl, bo0, bo1);
    }
  };
  if (kbase + KSL > kv_len) {
    auto bm = [&](int k) -> uint32_t { return k < kv_len ? 0xffu : 0u; };
    pv(bm(kq) | (bm(kq + 1) << 8) | (bm(kq + 8) << 16) | (bm(kq + 9) << 24),
       bm(kq + 16) | (bm(kq + 17) << 8) | (bm(kq + 24) << 16) | (bm(kq + 25) << 24));
  } else {
    pv(0xffffffffu, 0xffffffffu);
  }
}

// The decode role over an FP8 (E4M3) cache: the 16-bit role's item queue,
// stage ring and combine, with 128-key stages of one-byte codes, the item's
// Q rewritten as e4m3 parts and decode_stage_f8 for the products.
template <typename T, int D, bool F8, int LT, bool RP>
__device__ bool decode_role_f8(const PodParams& P, uint8_t* smem) {
  using L = DLayout<D, RP>;
  constexpr bool BF16 = Pack<T>::kBF16;
  constexpr int NKB = L::NKB;
  static_assert(F8 && L::F8OK && LT == POD_LT_NONE,
                "FP8 decode caches are built for head_dim 128 without a logits transform");
  // keys per stage and per warp (each m-tile's 4 warps split a stage's keys)
  constexpr int KST = L::F8_KEYS;
  constexpr int KSL = KST / 4;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int mt = warp >> 2, ks = warp & 3;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + L::BAR_OFF;   // full[NSTAGE]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::BAR_OFF + 64);
  const int G = P.G, H = P.H;
  T* __restrict__ outg = reinterpret_cast<T*>(P.out_d);
  const float NEG_INF = -INFINITY;
  volatile int* item_slot = reinterpret_cast<volatile int*>(smem + L::BAR_OFF + 96);

  if (tid == 0) {
    for (int s = 0; s < L::NSTAGE; ++s) mbar_init(bar0 + 8 * s, P.d_tma ? 1u : (uint32_t)kThreads);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (P.d_tma && tid == 0) {
    tma_prefetch_desc(&P.tm_kv_d);
    tma_prefetch_desc(&P.tm_q_d);
  }
  const uint32_t q_bytes = (uint32_t)(L::NQ * NKB * 128 * G * P.tu);
  int fills = 0;
  bool ok = true;

  for (;;) {
    // thread 0 takes the next queue position; its record carries everything
    // the item needs, so the claim costs one dependent load
    if (tid == 0) {
      const int idx = atomicAdd(P.status + 9, 1);
      *item_slot = idx < P.n_items ? idx : -1;
    }
    __syncthreads();
    const int pos = *item_slot;
    if (pos < 0 || !ok) break;
    const int32_t* rec = P.dqrec + POD_DQREC * pos;
    // CUDA-graph capacity mode: n_items is the capacity and the records past
    // the plan's own items have request -1 (the queue is empty there)
    if (rec[0] < 0) break;
    const int g = rec[1], tok0 = rec[2], ntok = rec[3], k0 = rec[4], k1 = rec[5];
    const int R = ntok * G;
    const int Mt = (R + 15) >> 4;
    const int kv_len = rec[8];
    const int q_base = rec[9];
    const int q_len = rec[10];
    const int page_base = rec[11];
    const int npages = rec[12];
    const int kb0 = (k0 / KST) * KST;
    const int nst = (k1 - kb0 + KST - 1) / KST;

    // TMA path: page of box `lane` of stage st (lane < KST / d_tma <= 16). A
    // box past the request's last page, or wholly outside [k0, k1) (the
    // 128-key stages overhang the 64-key chunk bounds), takes the
    // out-of-range page id, which TMA fills with zeros without reading HBM.
    auto page_for = [&](int st) -> int {
      const int t = kb0 + st * KST + lane * P.d_tma;
      const int pidx = t >> P.ps_shift;
      return (pidx < npages && t < k1 && t + P.d_tma > k0)
                 ? __ldg(P.d_kv_indices + page_base + pidx) : P.d_num_pages;
    };
    // fill stage st of this item (Q travels with stage 0) into ring slot
    // (fills + st) % 3; TMA path: `page` = page_for(st) of this lane, or -1
    // to look it up here
    auto issue = [&](int st, int page) {
      const int f = fills + st;
      const int buf = f % L::NSTAGE;
      const uint32_t full = bar0 + 8 * buf;
      const int kb = kb0 + st * KST;
      if (P.d_tma) {
        // warp 0: lane 0 registers the bytes, lane i fetches box group i
        if (warp == 0) {
          if (lane == 0) {
            mbar_arrive_expect_tx(full, (uint32_t)L::F8_STAGE + (st == 0 ? q_bytes : 0u));
            if (st == 0)
              for (int dh = 0; dh < NKB; ++dh)
                tma_load_3d(sbase + L::Q_OFF + dh * L::QDH, &P.tm_q_d, dh * 64, g * G, q_base + tok0,
                            full);
          }
          __syncwarp();
          if (lane < KST / P.d_tma) {
            // one-byte codes: a key's head row is one 128-byte row
            if (page < 0) page = page_for(st);
            const int o = lane * P.d_tma;
            const uint32_t k8 = sbase + L::STAGE_OFF + buf * L::F8_STAGE + (uint32_t)o * 128u;
            if (P.ps >= 8) {  // coordinates (x, slot, head, 2 * page + kv)
              const int tin = (kb + o) & (P.ps - 1);
              tma_load_4d(k8, &P.tm_kv_d, 0, tin, g, 2 * page, full);
              tma_load_4d(k8 + L::F8_HALF, &P.tm_kv_d, 0, tin, g, 2 * page + 1, full);
            } else {          // page_size 1: (x, page, head, kv)
              tma_load_4d(k8, &P.tm_kv_d, 0, page, g, 0, full);
              tma_load_4d(k8 + L::F8_HALF, &P.tm_kv_d, 0, page, g, 1, full);
            }
          }
        }
      } else {
        const T* __restrict__ qg = reinterpret_cast<const T*>(P.q_d);
        if (st == 0) {
          for (int idx = tid; idx < POD_DECODE_ROWS * (D / 8); idx += kThreads) {
            const int r = idx / (D / 8), c = idx % (D / 8);
            const bool valid = r < R;
            const int tok = tok0 + (valid ? r / G : 0);
            const int head = g * G + (valid ? r % G : 0);
            const size_t qoff = ((size_t)(q_base + tok) * H + head) * D + c * 8;
            cp_async16(sbase + L::Q_OFF + (c >> 3) * L::QDH + sw128_off(r, c & 7), qg + qoff,
                       valid ? 16u : 0u);
          }
        }
        // one-byte codes, [key][128 B] per K or V: 8 chunks of 16 B a key
        const uint8_t* __restrict__ kv8 = reinterpret_cast<const uint8_t*>(P.kv_d);
        const uint32_t k8 = sbase + L::STAGE_OFF + buf * L::F8_STAGE;
        const size_t vstride8 = (size_t)P.ps * P.Hk * D;
        constexpr int PER8 = KST * 8 / kThreads;
#pragma unroll 1
        for (int i = 0; i < PER8; ++i) {
          const int idx = tid + kThreads * i;
          const int key = idx >> 3, c = idx & 7;
          const int t = kb + key;
          const bool valid = t >= k0 && t < k1;
          const int tt = valid ? t : k0;
          const int pg = __ldg(P.d_kv_indices + page_base +
                               (P.ps_shift >= 0 ? (tt >> P.ps_shift) : (tt / P.ps)));
          const int slot = P.ps_shift >= 0 ? (tt & (P.ps - 1)) : (tt % P.ps);
          const uint8_t* src = kv8 + (P.d_hnd
              ? (((size_t)pg * 2 * P.Hk + g) * P.ps + slot) * D + c * 16
              : (((size_t)pg * 2 * P.ps + slot) * P.Hk + g) * D + c * 16);
          const uint32_t off = (uint32_t)key * 128u + (uint32_t)((c ^ (key & 7)) << 4);
          cp_async16(k8 + off, src, valid ? 16u : 0u);
          cp_async16(k8 + L::F8_HALF + off, src + vstride8, valid ? 16u : 0u);
        }
        cp_async_mbar_arrive(full);
      }
    };
    const int npre = nst < L::NSTAGE ? nst : L::NSTAGE;
    for (int st = 0; st < npre; ++st) issue(st, -1);

    if (nst > 0) {
      // wait for stage 0 here (the stage loop's own wait then passes at once),
      // before the accumulators are live
      const bool got = __all_sync(
          0xffffffffu,
          mbar_wait(bar0 + 8 * (fills % L::NSTAGE), (fills / L::NSTAGE) & 1, abort_flag));
      // Q landed with stage 0: rewrite it as NP e4m3 parts. Row r is first
      // scaled by 2^e (e puts its largest |q| in [128, 256)); part p holds
      // the E4M3 rounding of what parts 0..p-1 left, so the parts sum to
      // the scaled row: exactly for bf16 (8 bits in two parts of 4) and to
      // 12 bits for fp16 (three parts), down to 2^-9 of the scaled units.
      constexpr int NP = BF16 ? 2 : 3;
      const int row = tid >> 3, seg = tid & 7;   // 16 elements: d 16 seg ..
      float x[16];
      float mxq = 0.f;
      {
        const int dh = seg >> 2, c0 = 2 * (seg & 3);
        const uint32_t ra = sbase + L::Q_OFF + dh * L::QDH + row * 128;
        uint32_t w[8];
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "r"(ra + ((c0 ^ (row & 7)) << 4)));
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
                     : "r"(ra + (((c0 + 1) ^ (row & 7)) << 4)));
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float2 v = Pack<T>::unpack(w[i]);
          x[2 * i] = v.x;
          x[2 * i + 1] = v.y;
          mxq = fmaxf(mxq, fmaxf(fabsf(v.x), fabsf(v.y)));
        }
      }
      mxq = fmaxf(mxq, __shfl_xor_sync(0xffffffffu, mxq, 1));
      mxq = fmaxf(mxq, __shfl_xor_sync(0xffffffffu, mxq, 2));
      mxq = fmaxf(mxq, __shfl_xor_sync(0xffffffffu, mxq, 4));
      const int eb = (int)((__float_as_uint(mxq) >> 23) & 0xffu);  // biased exponent
      const int e = mxq > 0.f ? min(max(134 - eb, -120), 120) : 0;  // 7 - floor(log2)
      const float up = __uint_as_float((uint32_t)(127 + e) << 23);
      uint32_t part[NP][4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float v[4] = {x[4 * i] * up, x[4 * i + 1] * up, x[4 * i + 2] * up, x[4 * i + 3] * up};
#pragma unroll
        for (int pp = 0; pp < NP; ++pp) {
          const uint32_t h01 = f32x2_to_e4m3x2(v[0], v[1]), h23 = f32x2_to_e4m3x2(v[2], v[3]);
          part[pp][i] = h01 | (h23 << 16);
          if (pp + 1 < NP) {
            const uint32_t f01 = e4m3x2_to<__half>((uint16_t)h01);
            const uint32_t f23 = e4m3x2_to<__half>((uint16_t)h23);
            const float2 g01 = __half22float2(*reinterpret_cast<const __half2*>(&f01));
            const float2 g23 = __half22float2(*reinterpret_cast<const __half2*>(&f23));
            v[0] -= g01.x;
            v[1] -= g01.y;
            v[2] -= g23.x;
            v[3] -= g23.y;
          }
        }
      }
      __syncthreads();  // every 16-bit Q element is read before parts 0-1 overwrite them
      if (got) {
#pragma unroll
        for (int pp = 0; pp < NP; ++pp) {
          const uint32_t dst = sbase + (pp < 2 ? L::Q_OFF + pp * L::Q8_PART : L::Q8X_OFF) +
                               row * 128 + ((seg ^ (row & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(part[pp][0]),
                       "r"(part[pp][1]), "r"(part[pp][2]), "r"(part[pp][3]) : "memory");
        }
        if (seg == 0) {
          // row info for the stages: key range [lo, hi) and the softmax scale with 2^-e
          const int tok = tok0 + (row < R ? row / G : 0);
          const int pd = kv_len - q_len + tok;
          int4 ri;
          ri.x = max(P.window_left >= 0 ? max(pd - P.window_left, 0) : 0, k0);
          ri.y = min(P.causal ? min(pd + 1, kv_len) : kv_len, k1);
          ri.z = (int)__float_as_uint(P.d_scale_log2 * __uint_as_float((uint32_t)(127 - e) << 23));
          ri.w = 0;
          asm volatile("st.shared.v4.s32 [%0], {%1, %2, %3, %4};" ::"r"(sbase + L::QSC_OFF + row * 16),
                       "r"(ri.x), "r"(ri.y), "r"(ri.z), "r"(ri.w) : "memory");
        }
      }
      __syncthreads();
    }
    float m[2] = {NEG_INF, NEG_INF}, l[2] = {0.f, 0.f};
    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    const bool active = mt < Mt;

    for (int st = 0; st < nst; ++st) {
      const int f = fills + st;
      const int buf = f % L::NSTAGE;
      // look up the pages of the stage this one's slot is refilled with now, so
      // that the load latency hides behind the compute
      const int next_page =
          (P.d_tma && warp == 0 && st + L::NSTAGE < nst) ? page_for(st + L::NSTAGE) : -1;
      // warp-uniform, so that every lane reaches the warp votes of its stage
      const bool got =
          __all_sync(0xffffffffu, mbar_wait(bar0 + 8 * buf, (f / L::NSTAGE) & 1, abort_flag));
      const int kbase = kb0 + st * KST + ks * KSL;
      if (got && active && kbase < k1 && kbase + KSL > k0)
        decode_stage_f8<BF16, D, KSL>(sbase + L::STAGE_OFF + buf * L::F8_STAGE, L::F8_HALF,
                                      sbase + L::Q_OFF, L::Q8_PART, sbase + L::Q8X_OFF, mt, ks,
                                      lane, kbase, kv_len, sbase + L::QSC_OFF, m, l, o);
      if (!__syncthreads_and(got)) { ok = false; break; }
      if (st + L::NSTAGE < nst) issue(st + L::NSTAGE, next_page);
    }
    fills += nst;
    if (!ok) break;

    // ---- combine the 4 key slices of each m-tile through shared memory
    // (the output placement is read from the record again rather than kept
    // live in registers across the stage loop)
    const int32_t* crec = P.dqrec + POD_DQREC * pos;
    const int cg = __ldg(crec + 1), ctok0 = __ldg(crec + 2), prow = __ldg(crec + 6);
    const int cq_base = __ldg(crec + 9);
    float* scr_o = reinterpret_cast<float*>(smem + L::SCR_O);
    float* scr_ml = reinterpret_cast<float*>(smem + L::SCR_ML);
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      l[h2] += __shfl_xor_sync(0xffffffffu, l[h2], 1);
      l[h2] += __shfl_xor_sync(0xffffffffu, l[h2], 2);
    }
    if (active) {
      float* wo = scr_o + warp * 16 * D;
      const int rl = lane >> 2;
      // d 16q + 4t .. +3 from the even / odd tiles of chunk q
#pragma unroll
      for (int q = 0; q < D / 16; ++q) {
        const int col = 16 * q + 4 * (lane & 3);
        *reinterpret_cast<float4*>(wo + rl * D + col) =
            make_float4(o[2 * q][0], o[2 * q + 1][0], o[2 * q][1], o[2 * q + 1][1]);
        *reinterpret_cast<float4*>(wo + (rl + 8) * D + col) =
            make_float4(o[2 * q][2], o[2 * q + 1][2], o[2 * q][3], o[2 * q + 1][3]);
      }
      if ((lane & 3) == 0) {
        const int rl = lane >> 2;
        scr_ml[(warp * 16 + rl) * 2 + 0] = m[0];
        scr_ml[(warp * 16 + rl) * 2 + 1] = l[0];
        scr_ml[(warp * 16 + rl + 8) * 2 + 0] = m[1];
        scr_ml[(warp * 16 + rl + 8) * 2 + 1] = l[1];
      }
    }
    __syncthreads();
    for (int idx = tid; idx < R * (D / 4); idx += kThreads) {
      const int rr = idx / (D / 4), c4 = (idx % (D / 4)) * 4;
      const int mtr = rr >> 4, rl = rr & 15;
      float M = NEG_INF;
#pragma unroll
      for (int k = 0; k < 4; ++k) M = fmaxf(M, scr_ml[((mtr * 4 + k) * 16 + rl) * 2]);
      const float Ms = (M == NEG_INF) ? 0.f : M;
      float wsum = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int wk = mtr * 4 + k;
        const float wgt = ex2(scr_ml[(wk * 16 + rl) * 2] - Ms);
        wsum += wgt * scr_ml[(wk * 16 + rl) * 2 + 1];
        const float4 v = *reinterpret_cast<const float4*>(scr_o + (wk * 16 + rl) * D + c4);
        acc.x += wgt * v.x;
        acc.y += wgt * v.y;
        acc.z += wgt * v.z;
        acc.w += wgt * v.w;
      }
      const int tok = ctok0 + rr / G;
      const int head = cg * G + rr % G;
      // the slices carried 256 P (sums and outputs)
      constexpr float kPU = 1.f / 256.f;
      wsum *= kPU;
      if (prow < 0) {
        float denom = wsum;
        if (P.has_sinks) denom += ex2(P.sinks[head] * 1.4426950408889634f - Ms);
        const float inv = denom > 0.f ? P.v_scale * kPU / denom : 0.f;
        const size_t orow = (size_t)(cq_base + tok) * H + head;
        uint2 v;
        v.x = Pack<T>::two(acc.x * inv, acc.y * inv);
        v.y = Pack<T>::two(acc.z * inv, acc.w * inv);
        *reinterpret_cast<uint2*>(outg + orow * D + c4) = v;
        if (c4 == 0 && P.lse_d) P.lse_d[orow] = wsum > 0.f ? M + log2f(wsum) : NEG_INF;
      } else {
        const float inv = wsum > 0.f ? P.v_scale * kPU / wsum : 0.f;
        *reinterpret_cast<float4*>(P.part_o + (size_t)(prow + rr) * D + c4) =
            make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        if (c4 == 0) P.part_lse[prow + rr] = wsum > 0.f ? M + log2f(wsum) : NEG_INF;
      }
    }
    // the combine's generic accesses to the stage area come before the next
    // item's TMA writes into it (stage reads within an item are ordered by the
    // per-stage barrier)
    fence_proxy_async();
    __syncthreads();
  }
  if (!ok) {
    *abort_flag = 1;
    if (tid == 0) raise_status(P.status, POD_STATUS_TIMEOUT);
  }
  cp_async_wait_all();
  if (ok && tid == 0)  // every filled stage was waited on: no transfer is pending
    for (int s = 0; s < L::NSTAGE; ++s) mbar_inval(bar0 + 8 * s);
  return ok;
}

template <typename T, int D, bool F8, int LT, bool RP>
__device__ bool decode_role(const PodParams& P, uint8_t* smem) {
  static_assert(!F8, "FP8 decode caches run decode_role_f8");  // 16-bit caches
  using L = DLayout<D, RP>;
  constexpr bool BF16 = Pack<T>::kBF16;
  constexpr int NKB = L::NKB;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int mt = warp >> 2, ks = warp & 3;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + L::BAR_OFF;   // full[NSTAGE]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::BAR_OFF + 64);
  const int G = P.G, H = P.H;
  T* __restrict__ outg = reinterpret_cast<T*>(P.out_d);
  const float NEG_INF = -INFINITY;
  volatile int* item_slot = reinterpret_cast<volatile int*>(smem + L::BAR_OFF + 96);

  if (tid == 0) {
    for (int s = 0; s < L::NSTAGE; ++s) mbar_init(bar0 + 8 * s, P.d_tma ? 1u : (uint32_t)kThreads);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (P.d_tma && tid == 0) {
    tma_prefetch_desc(&P.tm_kv_d);
    tma_prefetch_desc(&P.tm_q_d);
  }
  const uint32_t q_bytes = (uint32_t)(L::NQ * NKB * 128 * G * P.tu);
  // K/V stage layout: [key / kbx][d half][key % kbx][64 elements] in 128-byte
  // swizzled rows, kbx = keys per TMA box (64 on the cp.async path, where it
  // is [d half][key][64]). Row offset of key k in its d half 0:
  const int kshift = P.d_tma ? 31 - __clz(P.d_tma) : 6;
  const uint32_t half_stride = 128u << kshift;  // bytes between the d halves of a box
  auto key_row = [&](int k) -> uint32_t {
    return (uint32_t)((k >> kshift) << kshift) * (NKB * 128u) +
           (uint32_t)(k & ((1 << kshift) - 1)) * 128u;
  };
  int fills = 0;
  bool ok = true;

  for (;;) {
    // thread 0 takes the next queue position; its record carries everything
    // the item needs, so the claim costs one dependent load
    if (tid == 0) {
      const int idx = atomicAdd(P.status + 9, 1);
      *item_slot = idx < P.n_items ? idx : -1;
    }
    __syncthreads();
    const int pos = *item_slot;
    if (pos < 0 || !ok) break;
    const int32_t* rec = P.dqrec + POD_DQREC * pos;
    // CUDA-graph capacity mode: n_items is the capacity and the records past
    // the plan's own items have request -1 (the queue is empty there)
    if (rec[0] < 0) break;
    const int g = rec[1], tok0 = rec[2], ntok = rec[3], k0 = rec[4], k1 = rec[5];
    const int R = ntok * G;
    const int Mt = (R + 15) >> 4;
    const int kv_len = rec[8];
    const int q_base = rec[9];
    const int q_len = rec[10];
    const int page_base = rec[11];
    const int npages = rec[12];
    const int kb0 = (k0 / POD_DECODE_STAGE) * POD_DECODE_STAGE;
    const int nst = (k1 - kb0 + POD_DECODE_STAGE - 1) / POD_DECODE_STAGE;

    // TMA path: page of box `lane` of stage st (lane < 64 / d_tma <= 8); an id
    // past the request's last page is the out-of-range page TMA fills with zeros
    auto page_for = [&](int st) -> int {
      const int pidx = (kb0 + st * POD_DECODE_STAGE + lane * P.d_tma) >> P.ps_shift;
      return pidx < npages ? __ldg(P.d_kv_indices + page_base + pidx) : P.d_num_pages;
    };
    // fill stage st of this item (Q travels with stage 0) into ring slot
    // (fills + st) % 3; TMA path: `page` = page_for(st) of this lane, or -1
    // to look it up here
    auto issue = [&](int st, int page) {
      const int f = fills + st;
      const int buf = f % L::NSTAGE;
      const uint32_t full = bar0 + 8 * buf;
      const uint32_t sk = sbase + L::STAGE_OFF + buf * L::STAGE_BYTES;
      const uint32_t sv = sk + L::KBYTES;
      const int kb = kb0 + st * POD_DECODE_STAGE;
      if (P.d_tma) {
        // warp 0: lane 0 registers the bytes, lane i fetches box group i
        if (warp == 0) {
          if (lane == 0) {
            mbar_arrive_expect_tx(full, 2u * L::KBYTES +
                                            (st == 0 ? q_bytes : 0u));
            if (st == 0)
              for (int dh = 0; dh < NKB; ++dh) {
                tma_load_3d(sbase + L::Q_OFF + dh * L::QDH, &P.tm_q_d, dh * 64, g * G, q_base + tok0,
                            full);
                if (RP)
                  tma_load_3d(sbase + L::QLO_OFF + dh * L::QDH, &P.tm_qlo_d, dh * 64, g * G,
                              q_base + tok0, full);
              }
          }
          __syncwarp();
          if (lane < POD_DECODE_STAGE / P.d_tma) {
            if (page < 0) page = page_for(st);
            const int o = lane * P.d_tma;
            const uint32_t dst = (uint32_t)o * (NKB * 128u);
            if (P.ps >= 8) {  // coordinates (x, slot, half, head, 2 * page + kv)
              const int tin = (kb + o) & (P.ps - 1);
              tma_load_5d(sk + dst, &P.tm_kv_d, 0, tin, 0, g, 2 * page, full);
              tma_load_5d(sv + dst, &P.tm_kv_d, 0, tin, 0, g, 2 * page + 1, full);
            } else {          // page_size 1: (x, page, half, head, kv)
              tma_load_5d(sk + dst, &P.tm_kv_d, 0, page, 0, g, 0, full);
              tma_load_5d(sv + dst, &P.tm_kv_d, 0, page, 0, g, 1, full);
            }
          }
        }
      } else {
        const T* __restrict__ qg = reinterpret_cast<const T*>(P.q_d);
        const T* __restrict__ kvg = reinterpret_cast<const T*>(P.kv_d);
        if (st == 0) {
          for (int idx = tid; idx < POD_DECODE_ROWS * (D / 8); idx += kThreads) {
            const int r = idx / (D / 8), c = idx % (D / 8);
            const bool valid = r < R;
            const int tok = tok0 + (valid ? r / G : 0);
            const int head = g * G + (valid ? r % G : 0);
            const size_t qoff = ((size_t)(q_base + tok) * H + head) * D + c * 8;
            cp_async16(sbase + L::Q_OFF + (c >> 3) * L::QDH + sw128_off(r, c & 7), qg + qoff,
                       valid ? 16u : 0u);
            if (RP)
              cp_async16(sbase + L::QLO_OFF + (c >> 3) * L::QDH + sw128_off(r, c & 7),
                         reinterpret_cast<const T*>(P.q_d_lo) + qoff, valid ? 16u : 0u);
          }
        }
        constexpr int CH = POD_DECODE_STAGE * (D / 8);
        constexpr int PER = CH / kThreads;
        static_assert(CH % kThreads == 0, "stage chunks must divide evenly");
        int pages[PER];
#pragma unroll
        for (int i = 0; i < PER; ++i) {
          const int key = (tid + kThreads * i) / (D / 8);
          const int t = kb + key;
          const int tt = (t >= k0 && t < k1) ? t : k0;
          const int pg_i = P.ps_shift >= 0 ? (tt >> P.ps_shift) : (tt / P.ps);
          pages[i] = __ldg(P.d_kv_indices + page_base + pg_i);
        }
        const size_t vstride = (size_t)P.ps * P.Hk * D;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
          const int idx = tid + kThreads * i;
          const int key = idx / (D / 8), c = idx % (D / 8);
          const int t = kb + key;
          const bool valid = t >= k0 && t < k1;
          const int tt = valid ? t : k0;
          const int slot = P.ps_shift >= 0 ? (tt & (P.ps - 1)) : (tt % P.ps);
          const T* src = kvg + (P.d_hnd
              ? (((size_t)pages[i] * 2 * P.Hk + g) * P.ps + slot) * D + c * 8
              : (((size_t)pages[i] * 2 * P.ps + slot) * P.Hk + g) * D + c * 8);
          const uint32_t off = (c >> 3) * L::KDH + sw128_off(key, c & 7);
          cp_async16(sk + off, src, valid ? 16u : 0u);
          cp_async16(sv + off, src + vstride, valid ? 16u : 0u);
        }
        cp_async_mbar_arrive(full);
      }
    };
    const int npre = nst < L::NSTAGE ? nst : L::NSTAGE;
    for (int st = 0; st < npre; ++st) issue(st, -1);

    // rows of this thread inside its m-tile: r0 = 16 mt + lane/4, r1 = r0 + 8
    int row_lo[2], row_hi[2];
    // ALiBi only: the rows' slopes (raw q.k units) and diagonal positions
    float a_slope[2] = {0.f, 0.f};
    int a_pd[2] = {0, 0};
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      const int rr = mt * 16 + (lane >> 2) + 8 * h2;
      const int tok = tok0 + (rr < R ? rr / G : 0);
      const int pd = kv_len - q_len + tok;
      row_hi[h2] = min(P.causal ? min(pd + 1, kv_len) : kv_len, k1);
      row_lo[h2] = max(P.window_left >= 0 ? max(pd - P.window_left, 0) : 0, k0);
      if constexpr (LT == POD_LT_ALIBI) {
        a_slope[h2] = __ldg(P.alibi + g * G + (rr < R ? rr % G : 0)) * P.lt_inv_scale;
        a_pd[h2] = pd;
      }
    }
    float m[2] = {NEG_INF, NEG_INF}, l[2] = {0.f, 0.f};
    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    const bool active = mt < Mt;
    const int mi = lane >> 3;

    for (int st = 0; st < nst; ++st) {
      const int f = fills + st;
      const int buf = f % L::NSTAGE;
      // look up the pages of the stage this one's slot is refilled with now, so
      // that the load latency hides behind the compute
      const int next_page =
          (P.d_tma && warp == 0 && st + L::NSTAGE < nst) ? page_for(st + L::NSTAGE) : -1;
      const bool got = mbar_wait(bar0 + 8 * buf, (f / L::NSTAGE) & 1, abort_flag);
      // K of the stage (V follows at +KBYTES)
      const uint32_t sk = sbase + L::STAGE_OFF + buf * L::STAGE_BYTES;
      const int kbase = kb0 + st * POD_DECODE_STAGE + ks * 16;
      if (got && active && kbase < k1 && kbase + 16 > k0) {
        const uint32_t sq = sbase + L::Q_OFF;
        const uint32_t sv = sk + (uint32_t)L::KBYTES;
        float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
        if constexpr (RP) {
          // Keys rotated in registers: chunk kk (d 16kk..) pairs with chunk
          // kk + D/32 (d + D/2). A thread holds, for its keys ka (b[0], b[1])
          // and ka + 8 (b[2], b[3]), elements j = 16kk + 2(lane%4) + {0, 1}
          // (b[0], b[2]) and j + 8 (b[1], b[3]) of both chunks; each pair turns
          // by the angle of (key, j) from the cos/sin table (fp32 values of fp64
          // sincos), then splits into 16-bit high and low parts.
          constexpr int NC = D / 32;
          const int ta = min(kbase + (lane >> 2), P.rope_rows - 1);
          const int tb = min(kbase + 8 + (lane >> 2), P.rope_rows - 1);
          const float4* tra = reinterpret_cast<const float4*>(P.rope_tab + (size_t)ta * (D / 2));
          const float4* trb = reinterpret_cast<const float4*>(P.rope_tab + (size_t)tb * (D / 2));
#pragma unroll
          for (int kk = 0; kk < NC; ++kk) {
            uint32_t bx[4], by[4];
            {
              const int key = ks * 16 + (lane & 7) + ((mi >> 1) << 3);
              const int c0 = kk * 2 + (mi & 1), c1 = (kk + NC) * 2 + (mi & 1);
              ldsm_x4(sk + key_row(key) + (c0 >> 3) * half_stride + (((c0 & 7) ^ (lane & 7)) << 4),
                      bx[0], bx[1], bx[2], bx[3]);
              ldsm_x4(sk + key_row(key) + (c1 >> 3) * half_stride + (((c1 & 7) ^ (lane & 7)) << 4),
                      by[0], by[1], by[2], by[3]);
            }
            const float4 cs[4] = {__ldg(tra + 8 * kk + (lane & 3)), __ldg(tra + 8 * kk + 4 + (lane & 3)),
                                  __ldg(trb + 8 * kk + (lane & 3)), __ldg(trb + 8 * kk + 4 + (lane & 3))};
            uint32_t xh[4], xl[4], yh[4], yl[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 x = Pack<T>::unpack(bx[i]), y = Pack<T>::unpack(by[i]);
              const float x0 = fmaf(x.x, cs[i].x, -y.x * cs[i].y), y0 = fmaf(y.x, cs[i].x, x.x * cs[i].y);
              const float x1 = fmaf(x.y, cs[i].z, -y.y * cs[i].w), y1 = fmaf(y.y, cs[i].z, x.y * cs[i].w);
              Pack<T>::split(x0, x1, xh[i], xl[i]);
              Pack<T>::split(y0, y1, yh[i], yl[i]);
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int c = (kk + h * NC) * 2 + (mi >> 1);
              const int rr = mt * 16 + (lane & 7) + ((mi & 1) << 3);
              uint32_t ah[4], al[4];
              ldsm_x4(sq + (c >> 3) * L::QDH + sw128_off(rr, c & 7), ah[0], ah[1], ah[2], ah[3]);
              ldsm_x4(sq + (L::QLO_OFF - L::Q_OFF) + (c >> 3) * L::QDH + sw128_off(rr, c & 7), al[0],
                      al[1], al[2], al[3]);
              const uint32_t* bh = h ? yh : xh;
              const uint32_t* bl = h ? yl : xl;
              mma16816<BF16>(s0, ah, bh[0], bh[1]);
              mma16816<BF16>(s0, ah, bl[0], bl[1]);
              mma16816<BF16>(s0, al, bh[0], bh[1]);
              mma16816<BF16>(s1, ah, bh[2], bh[3]);
              mma16816<BF16>(s1, ah, bl[2], bl[3]);
              mma16816<BF16>(s1, al, bh[2], bh[3]);
            }
          }
        } else {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            uint32_t a[4], b[4];
            {
              const int rr = mt * 16 + (lane & 7) + ((mi & 1) << 3);
              const int c = kk * 2 + (mi >> 1);
              ldsm_x4(sq + (c >> 3) * L::QDH + sw128_off(rr, c & 7), a[0], a[1], a[2], a[3]);
            }
            {
              const int key = ks * 16 + (lane & 7) + ((mi >> 1) << 3);
              const int c = kk * 2 + (mi & 1);
              ldsm_x4(sk + key_row(key) + (c >> 3) * half_stride + (((c & 7) ^ (lane & 7)) << 4), b[0],
                      b[1], b[2], b[3]);
            }
            mma16816<BF16>(s0, a, b[0], b[1]);
            mma16816<BF16>(s1, a, b[2], b[3]);
          }
        }
        // mask, online softmax in base 2 (rows h2 = 0: c0,c1; h2 = 1: c2,c3)
        const int kq = kbase + 2 * (lane & 3);
        const float scale = P.d_scale_log2;  // sm_scale * log2(e)
        float mx[2];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          float* a0 = s0 + 2 * h2;
          float* a1 = s1 + 2 * h2;
          const int key[4] = {kq, kq + 1, kq + 8, kq + 9};
          float* v[4] = {a0, a0 + 1, a1, a1 + 1};
          float mm = NEG_INF;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float x = *v[e];
            if (LT == POD_LT_SOFTCAP || (RP && P.lt == POD_LT_SOFTCAP))
              x = soft_cap(x, P.lt_c, 1.f / P.lt_c);
            if constexpr (LT == POD_LT_ALIBI) x = fmaf(a_slope[h2], (float)(key[e] - a_pd[h2]), x);
            if (key[e] < row_lo[h2] || key[e] >= row_hi[h2]) x = NEG_INF;
            *v[e] = x;
            mm = fmaxf(mm, x);
          }
          mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, 1));
          mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, 2));
          mx[h2] = mm * scale;
        }
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const float m_new = fmaxf(m[h2], mx[h2]);
          const float m_sub = (m_new == NEG_INF) ? 0.f : m_new;
          const float alpha = ex2(m[h2] - m_sub);
          m[h2] = m_new;
          float* a0 = s0 + 2 * h2;
          float* a1 = s1 + 2 * h2;
          a0[0] = ex2(fmaf(a0[0], scale, -m_sub));
          a0[1] = ex2(fmaf(a0[1], scale, -m_sub));
          a1[0] = ex2(fmaf(a1[0], scale, -m_sub));
          a1[1] = ex2(fmaf(a1[1], scale, -m_sub));
          l[h2] = l[h2] * alpha + (a0[0] + a0[1] + a1[0] + a1[1]);
#pragma unroll
          for (int i = 0; i < D / 8; ++i) {
            o[i][2 * h2] *= alpha;
            o[i][2 * h2 + 1] *= alpha;
          }
        }
        // P <= 1 rounded to the plan's 16-bit type for the PV product
        uint32_t pa[4];
        pa[0] = Pack<T>::two(s0[0], s0[1]);
        pa[1] = Pack<T>::two(s0[2], s0[3]);
        pa[2] = Pack<T>::two(s1[0], s1[1]);
        pa[3] = Pack<T>::two(s1[2], s1[3]);
        // V rows at or past kv_len may be unused slots of the last page: zero
        // them in the fragments so that P = 0 never meets a non-finite value
        uint32_t vm0 = 0xffffffffu, vm1 = 0xffffffffu;
        if (kbase + 16 > kv_len) {
          vm0 = (kq < kv_len ? 0x0000ffffu : 0u) | (kq + 1 < kv_len ? 0xffff0000u : 0u);
          vm1 = (kq + 8 < kv_len ? 0x0000ffffu : 0u) | (kq + 9 < kv_len ? 0xffff0000u : 0u);
        }
#pragma unroll
        for (int j = 0; j < D / 16; ++j) {
          uint32_t b[4];
          const int key = ks * 16 + (lane & 7) + ((mi & 1) << 3);
          const int c = 2 * j + (mi >> 1);
          ldsm_x4_t(sv + key_row(key) + (c >> 3) * half_stride + (((c & 7) ^ (lane & 7)) << 4), b[0],
                    b[1], b[2], b[3]);
          mma16816<BF16>(o[2 * j], pa, b[0] & vm0, b[1] & vm1);
          mma16816<BF16>(o[2 * j + 1], pa, b[2] & vm0, b[3] & vm1);
        }
      }
      if (!__syncthreads_and(got)) { ok = false; break; }
      if (st + L::NSTAGE < nst) issue(st + L::NSTAGE, next_page);
    }
    fills += nst;
    if (!ok) break;

    // ---- combine the 4 key slices of each m-tile through shared memory
    // (the output placement is read from the record again rather than kept
    // live in registers across the stage loop)
    const int32_t* crec = P.dqrec + POD_DQREC * pos;
    const int cg = __ldg(crec + 1), ctok0 = __ldg(crec + 2), prow = __ldg(crec + 6);
    const int cq_base = __ldg(crec + 9);
    float* scr_o = reinterpret_cast<float*>(smem + L::SCR_O);
    float* scr_ml = reinterpret_cast<float*>(smem + L::SCR_ML);
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      l[h2] += __shfl_xor_sync(0xffffffffu, l[h2], 1);
      l[h2] += __shfl_xor_sync(0xffffffffu, l[h2], 2);
    }
    if (active) {
      float* wo = scr_o + warp * 16 * D;
      const int rl = lane >> 2;
#pragma unroll
      for (int i = 0; i < D / 8; ++i) {
        const int col = 8 * i + 2 * (lane & 3);
        *reinterpret_cast<float2*>(wo + rl * D + col) = make_float2(o[i][0], o[i][1]);
        *reinterpret_cast<float2*>(wo + (rl + 8) * D + col) = make_float2(o[i][2], o[i][3]);
      }
      if ((lane & 3) == 0) {
        const int rl = lane >> 2;
        scr_ml[(warp * 16 + rl) * 2 + 0] = m[0];
        scr_ml[(warp * 16 + rl) * 2 + 1] = l[0];
        scr_ml[(warp * 16 + rl + 8) * 2 + 0] = m[1];
        scr_ml[(warp * 16 + rl + 8) * 2 + 1] = l[1];
      }
    }
    __syncthreads();
    for (int idx = tid; idx < R * (D / 4); idx += kThreads) {
      const int rr = idx / (D / 4), c4 = (idx % (D / 4)) * 4;
      const int mtr = rr >> 4, rl = rr & 15;
      float M = NEG_INF;
#pragma unroll
      for (int k = 0; k < 4; ++k) M = fmaxf(M, scr_ml[((mtr * 4 + k) * 16 + rl) * 2]);
      const float Ms = (M == NEG_INF) ? 0.f : M;
      float wsum = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int wk = mtr * 4 + k;
        const float wgt = ex2(scr_ml[(wk * 16 + rl) * 2] - Ms);
        wsum += wgt * scr_ml[(wk * 16 + rl) * 2 + 1];
        const float4 v = *reinterpret_cast<const float4*>(scr_o + (wk * 16 + rl) * D + c4);
        acc.x += wgt * v.x;
        acc.y += wgt * v.y;
        acc.z += wgt * v.z;
        acc.w += wgt * v.w;
      }
      const int tok = ctok0 + rr / G;
      const int head = cg * G + rr % G;
      if (prow < 0) {
        float denom = wsum;
        if (P.has_sinks) denom += ex2(P.sinks[head] * 1.4426950408889634f - Ms);
        const float inv = denom > 0.f ? P.v_scale / denom : 0.f;
        const size_t orow = (size_t)(cq_base + tok) * H + head;
        uint2 v;
        v.x = Pack<T>::two(acc.x * inv, acc.y * inv);
        v.y = Pack<T>::two(acc.z * inv, acc.w * inv);
        *reinterpret_cast<uint2*>(outg + orow * D + c4) = v;
        if (c4 == 0 && P.lse_d) P.lse_d[orow] = wsum > 0.f ? M + log2f(wsum) : NEG_INF;
      } else {
        const float inv = wsum > 0.f ? P.v_scale / wsum : 0.f;
        *reinterpret_cast<float4*>(P.part_o + (size_t)(prow + rr) * D + c4) =
            make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        if (c4 == 0) P.part_lse[prow + rr] = wsum > 0.f ? M + log2f(wsum) : NEG_INF;
      }
    }
    // the combine's generic accesses to the stage area come before the next
    // item's TMA writes into it (stage reads within an item are ordered by the
    // per-stage barrier)
    fence_proxy_async();
    __syncthreads();
  }
  if (!ok) {
    *abort_flag = 1;
    if (tid == 0) raise_status(P.status, POD_STATUS_TIMEOUT);
  }
  cp_async_wait_all();
  if (ok && tid == 0)  // every filled stage was waited on: no transfer is pending
    for (int s = 0; s < L::NSTAGE; ++s) mbar_inval(bar0 + 8 * s);
  return ok;
}

template <typename T, int D, bool F8, int LT, bool RP>
__device__ __forceinline__ bool decode_dispatch(const PodParams& P, uint8_t* smem) {
  if constexpr (F8) return decode_role_f8<T, D, F8, LT, RP>(P, smem);
  else return decode_role<T, D, F8, LT, RP>(P, smem);
}

// ============================================================ kernels
// F8: the decode half reads an FP8 (E4M3) cache (head_dim 128 only).
// LT: logits transform of both halves (POD_LT_NONE, _SOFTCAP, _ALIBI).
// RP: ROPE_LLAMA (one CTA per SM; a soft cap is then a run-time switch).
template <typename T, int D, bool F8, int LT, bool RP>
__global__ void __launch_bounds__(kThreads, (ctas_per_sm<D, RP>()))
    pod_kernel(const __grid_constant__ PodParams P) {
  extern __shared__ __align__(1024) uint8_t smem[];
  // the merge kernel may start its prologue now; it waits for this grid's completion
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tid = threadIdx.x, warp = tid >> 5;
  bool aligned = (smem_u32(smem) & 1023u) == 0u;  // 128B-swizzle atoms need 1024-byte alignment
  if (!aligned) {
    if (tid == 0) raise_status(P.status, POD_STATUS_ALIGN);
  } else {
    // Every CTA holds 256 TMEM columns for its life (two CTAs fill an SM's
    // 512); giving up the allocation permit at once lets the second CTA in.
    const uint32_t tslot = smem_u32(smem) + PLayout<D, RP>::BAR_OFF + 224;
    if (warp == 4) {
      tmem_alloc(tslot, PLayout<D, RP>::TMEM_COLS);
      tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + PLayout<D, RP>::BAR_OFF + 224);
    // Both queues are drained by every CTA: its own role's queue first (the
    // plan sizes the split), then the other one, so whichever half finishes
    // early helps with the rest.
    const bool p_first = (int)blockIdx.x < P.n_p_ctas;
    bool ok = true;
    for (int phase = 0; phase < 2 && ok; ++phase) {
      const bool do_prefill = (phase == 0) == p_first;
      if (do_prefill ? P.n_tiles == 0 : P.n_items == 0) continue;
      // shared memory changes hands between the generic and the async proxy
      fence_proxy_async();
      __syncthreads();
      ok = do_prefill ? prefill_role<T, D, LT, RP>(P, smem, tmem)
                      : decode_dispatch<T, D, F8, LT, RP>(P, smem);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 4) tmem_dealloc(tmem, PLayout<D, RP>::TMEM_COLS);
  }
  // the last CTA to finish rewinds the queue counters for the next launch
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(P.status + 10, 1) == (int)gridDim.x - 1) {
      atomicExch(P.status + 8, 0);
      atomicExch(P.status + 9, 0);
      atomicExch(P.status + 10, 0);
    }
  }
}

// Launches K1 for one variant. The dynamic shared-memory attributes belong to
// each device's context: they are set once per device (and thread-safely).
template <typename T, int D, bool F8, int LT, bool RP>
cudaError_t launch_pod(const PodParams& P, cudaStream_t stream) {
  constexpr int SMEM = smem_bytes<D, RP, F8>();
  static std::atomic<unsigned long long> done{0ull};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
  if (bit == 0ull || !(done.load(std::memory_order_acquire) & bit)) {
    std::lock_guard<std::mutex> lock(mu);
    e = cudaFuncSetAttribute(pod_kernel<T, D, F8, LT, RP>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    // two CTAs per SM need the largest shared-memory carveout
    e = cudaFuncSetAttribute(pod_kernel<T, D, F8, LT, RP>,
                             cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    done.fetch_or(bit, std::memory_order_acq_rel);
  }
  pod_kernel<T, D, F8, LT, RP><<<P.grid, kThreads, SMEM, stream>>>(P);
  return cudaGetLastError();
}

}  // namespace
