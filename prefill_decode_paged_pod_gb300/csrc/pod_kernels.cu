// pod_kernels.cu — the fused POD launch for sm_103a and the split merge.
//
// K1 `pod_kernel`: one persistent grid; CTA c < n_prefill_ctas runs prefill
// tiles, the other CTAs run decode items (POD walkthrough, "POD 是什么": one
// launch serves the compute-bound prefill and the memory-bound decode, so the
// two share the SMs instead of leaving gaps between two launches).
//
//  prefill tile (128 query rows = ntok tokens x G qo heads of one KV head):
//    warps 5-7  cp.async loaders: Q tile once, then 64-key K/V blocks gathered
//               through the page table into two 128B-swizzled stages;
//    warp 4     one thread issues tcgen05.mma: S = Q K^T into TMEM (double
//               buffered), later O += P V into TMEM;
//    warps 0-3  one TMEM lane (= one query row) per thread: tcgen05.ld of S,
//               bottom-right causal / window mask, online softmax in base 2
//               with lazy rescaling of O, P written to shared memory as the
//               A operand of the next MMA, final O / (l + sink) and LSE.
//  decode item (<= 32 rows = q tokens x G heads, keys [k0, k1) of one chunk):
//    all 8 warps stream 64-key K/V stages with cp.async (3 stages); warp w
//    owns m-tile w/4 and keys 16*(w%4).. of each stage and runs mma.sync
//    m16n8k16 for Q K^T and P V with an online softmax in registers; warps
//    combine through shared memory and write the final output, or an fp32
//    partial (o, lse) when the plan split the KV range.
//
// K2 `pod_merge_kernel`: merges the split partials of each row with base-2
// LSE weights, adds the sink, writes out and LSE (flashinfer.cudnn page,
// "LSE 契约": base-2 LSE feeds a cascade merge). Launched with programmatic
// dependent launch; it waits on griddepcontrol.wait (POD walkthrough, "PDL").
#include <cuda_runtime.h>
#include <math.h>

#include "pod_device.cuh"
#include "pod_launch.h"
#include "pod_plan.h"

using namespace pod;

namespace {

constexpr int kThreads = 256;

// ------------------------------------------------------------------ layouts
template <int D>
struct PLayout {                                   // prefill shared memory
  static constexpr int NKB = D / 64;               // 64-element K blocks of head_dim
  static constexpr int QBLK = POD_TILE_ROWS * 128; // 128 rows x 128 B
  static constexpr int KVBLK = POD_KBLOCK * 128;   // 64 rows x 128 B
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + NKB * QBLK;
  static constexpr int V_OFF = K_OFF + 2 * NKB * KVBLK;
  static constexpr int P_OFF = V_OFF + 2 * NKB * KVBLK;
  static constexpr int BAR_OFF = P_OFF + POD_TILE_ROWS * 128;
  static constexpr int TOTAL = BAR_OFF + 256;
  static constexpr int TMEM_COLS = 256;            // S[2] (2 x 64) + O (<= 128)
  static constexpr int TM_S = 0, TM_O = 128;
};

template <int D>
struct DLayout {                                   // decode shared memory
  static constexpr int ROWB = D * 2;
  static constexpr int NCH = D / 8;
  static constexpr int KEYS = POD_DECODE_STAGE;
  static constexpr int Q_OFF = 0;
  static constexpr int STAGE_OFF = POD_DECODE_ROWS * ROWB;
  static constexpr int KBYTES = KEYS * ROWB;
  static constexpr int STAGE_BYTES = 2 * KBYTES;
  static constexpr int NSTAGE = 3;
  static constexpr int TOTAL = STAGE_OFF + NSTAGE * STAGE_BYTES;
  // combine scratch (reuses the stages): 8 warps x 16 rows x D floats, then m/l
  static constexpr int SCR_O = STAGE_OFF;
  static constexpr int SCR_ML = STAGE_OFF + 8 * 16 * D * 4;
  static_assert(SCR_ML + 8 * 16 * 2 * 4 <= TOTAL, "combine scratch must fit in the stages");
};

template <int D>
constexpr int smem_bytes() {
  return PLayout<D>::TOTAL > DLayout<D>::TOTAL ? PLayout<D>::TOTAL : DLayout<D>::TOTAL;
}

POD_DEV void raise_status(int32_t* status, int code) { atomicOr(status, code); }

// All 32 lanes wait; the result is warp-uniform so that warp-collective
// tcgen05.ld / __any_sync calls after it are reached by every lane.
POD_DEV bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  const bool ok = mbar_wait(bar, parity, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// ============================================================ prefill role
enum {
  B_QFULL = 0, B_QEMPTY = 1, B_KVFULL = 2, B_KVEMPTY = 4, B_SFULL = 6, B_SEMPTY = 8,
  B_PFULL = 10, B_PVDONE = 11, B_FINAL = 12
};

template <typename T, int D>
__device__ void prefill_role(const PodParams& P, uint8_t* smem, int cta) {
  using L = PLayout<D>;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + L::BAR_OFF;
  auto BAR = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::BAR_OFF + 128);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::BAR_OFF + 132);

  if (tid == 0) {
    mbar_init(BAR(B_QFULL), 96);
    mbar_init(BAR(B_QEMPTY), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(BAR(B_KVFULL + s), 96);
      mbar_init(BAR(B_KVEMPTY + s), 1);
      mbar_init(BAR(B_SFULL + s), 1);
      mbar_init(BAR(B_SEMPTY + s), 128);
    }
    mbar_init(BAR(B_PFULL), 128);
    mbar_init(BAR(B_PVDONE), 1);
    mbar_init(BAR(B_FINAL), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 4) {
    tmem_alloc(smem_u32(tmem_slot), L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int w_begin = P.cta_ptr[cta], w_end = P.cta_ptr[cta + 1];
  const int G = P.G, H = P.H;

  if (warp >= 5) {
    // ------------------------------------------------------------ loaders
    const int lt = tid - 160;  // 0..95
    const T* __restrict__ qg = reinterpret_cast<const T*>(P.q_p);
    const T* __restrict__ kvg = reinterpret_cast<const T*>(P.kv_p);
    int kv_fill = 0, q_fill = 0;
    bool ok = true;
    for (int w = w_begin; w < w_end && ok; ++w) {
      const int32_t* rec = P.ptiles + POD_REC * P.cta_list[w];
      const int req = rec[0], g = rec[1], tok0 = rec[2], ntok = rec[3], lo = rec[4], hi = rec[5];
      const int q_base = P.p_q_indptr[req];
      const int page_base = P.p_kv_indptr[req];
      const int nrows = ntok * G;
      if (!mbar_wait(BAR(B_QEMPTY), (q_fill & 1) ^ 1, abort_flag)) { ok = false; break; }
      constexpr int QCH = POD_TILE_ROWS * (D / 8);
      for (int idx = lt; idx < QCH; idx += 96) {
        const int r = idx / (D / 8), c = idx % (D / 8);
        const bool valid = r < nrows;
        const int tok = valid ? tok0 + r / G : tok0;
        const int head = valid ? g * G + r % G : g * G;
        const T* src = qg + ((size_t)(q_base + tok) * H + head) * D + c * 8;
        const uint32_t dst = sbase + L::Q_OFF + (c >> 3) * L::QBLK + sw128_off(r, c & 7);
        cp_async16(dst, src, valid ? 16u : 0u);
      }
      cp_async_mbar_arrive(BAR(B_QFULL));
      ++q_fill;
      const int b0 = (lo / POD_KBLOCK) * POD_KBLOCK;
      for (int kb = b0; kb < hi; kb += POD_KBLOCK) {
        const int s = kv_fill & 1;
        if (!mbar_wait(BAR(B_KVEMPTY + s), ((kv_fill >> 1) & 1) ^ 1, abort_flag)) { ok = false; break; }
        constexpr int KCH = POD_KBLOCK * (D / 8);
        for (int idx = lt; idx < 2 * KCH; idx += 96) {
          const int kv = idx / KCH, rem = idx % KCH;
          const int key = rem / (D / 8), c = rem % (D / 8);
          const int t = kb + key;
          const bool valid = t < hi;
          const int tt = valid ? t : kb;
          const int pg_i = P.ps_shift >= 0 ? (tt >> P.ps_shift) : (tt / P.ps);
          const int slot = P.ps_shift >= 0 ? (tt & (P.ps - 1)) : (tt % P.ps);
          const int page = __ldg(P.p_kv_indices + page_base + pg_i);
          const T* src = kvg + ((((size_t)page * 2 + kv) * P.ps + slot) * P.Hk + g) * D + c * 8;
          const uint32_t base = sbase + (kv ? L::V_OFF : L::K_OFF) + s * (L::NKB * L::KVBLK);
          const uint32_t dst = base + (c >> 3) * L::KVBLK + sw128_off(key, c & 7);
          cp_async16(dst, src, valid ? 16u : 0u);
        }
        cp_async_mbar_arrive(BAR(B_KVFULL + s));
        ++kv_fill;
      }
    }
    if (!ok) {
      *abort_flag = 1;
      raise_status(P.status, POD_STATUS_TIMEOUT);
    }
    cp_async_wait_all();
  } else if (warp == 4) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const bool bf16 = Pack<T>::kBF16;
      const uint32_t id_qk = idesc_f16(bf16, 128, POD_KBLOCK, false, false);
      const uint32_t id_pv = idesc_f16(bf16, 128, D, false, true);
      int kv_fill = 0, q_fill = 0, s_cnt = 0, p_cnt = 0;
      bool ok = true;
      for (int w = w_begin; w < w_end && ok; ++w) {
        const int32_t* rec = P.ptiles + POD_REC * P.cta_list[w];
        const int lo = rec[4], hi = rec[5];
        const int b0 = (lo / POD_KBLOCK) * POD_KBLOCK;
        const int nb = (hi - b0 + POD_KBLOCK - 1) / POD_KBLOCK;
        if (!mbar_wait(BAR(B_QFULL), q_fill & 1, abort_flag)) { ok = false; break; }
        ++q_fill;
        for (int j = 0; j <= nb && ok; ++j) {
          if (j < nb) {
            const int f = kv_fill + j;
            const int s = f & 1;
            if (!mbar_wait(BAR(B_KVFULL + s), (f >> 1) & 1, abort_flag)) { ok = false; break; }
            const int sc = s_cnt + j;
            const int b = sc & 1;
            if (!mbar_wait(BAR(B_SEMPTY + b), ((sc >> 1) & 1) ^ 1, abort_flag)) { ok = false; break; }
            tc_fence_after();
            fence_proxy_async();
            const uint32_t qa = sbase + L::Q_OFF;
            const uint32_t ka = sbase + L::K_OFF + s * (L::NKB * L::KVBLK);
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
              const uint64_t ad = sdesc_sw128(qa + (k >> 2) * L::QBLK + (k & 3) * 32, 16, 1024);
              const uint64_t bd = sdesc_sw128(ka + (k >> 2) * L::KVBLK + (k & 3) * 32, 16, 1024);
              mma_f16_ss(tmem + L::TM_S + b * POD_KBLOCK, ad, bd, id_qk, k > 0 ? 1u : 0u);
            }
            mma_commit(BAR(B_SFULL + b));
            if (j == nb - 1) mma_commit(BAR(B_QEMPTY));
          }
          if (j > 0) {
            // O += P_{j-1} V_{j-1}
            if (!mbar_wait(BAR(B_PFULL), p_cnt & 1, abort_flag)) { ok = false; break; }
            ++p_cnt;
            tc_fence_after();
            fence_proxy_async();
            const int s = (kv_fill + j - 1) & 1;
            const uint32_t pa = sbase + L::P_OFF;
            const uint32_t va = sbase + L::V_OFF + s * (L::NKB * L::KVBLK);
#pragma unroll
            for (int k = 0; k < POD_KBLOCK / 16; ++k) {
              const uint64_t ad = sdesc_sw128(pa + k * 32, 16, 1024);
              const uint64_t bd = sdesc_sw128(va + k * 2048, L::KVBLK, 1024);
              mma_f16_ss(tmem + L::TM_O, ad, bd, id_pv, (j > 1 || k > 0) ? 1u : 0u);
            }
            mma_commit(BAR(B_PVDONE));
            mma_commit(BAR(B_KVEMPTY + s));
          }
        }
        kv_fill += nb;
        s_cnt += nb;
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
    int s_cnt = 0, pv_cnt = 0;
    bool ok = true;
    const float NEG_INF = -INFINITY;
    for (int w = w_begin; w < w_end && ok; ++w) {
      const int32_t* rec = P.ptiles + POD_REC * P.cta_list[w];
      const int req = rec[0], g = rec[1], tok0 = rec[2], ntok = rec[3], lo = rec[4], hi = rec[5];
      const int prow = rec[6];
      const int kv_len = P.p_kv_len[req];
      const int q_len = P.p_q_indptr[req + 1] - P.p_q_indptr[req];
      const int nrows = ntok * G;
      const bool valid = r < nrows;
      const int tok = tok0 + (valid ? r / G : ntok - 1);
      const int head = g * G + (valid ? r % G : 0);
      const int pdiag = kv_len - q_len + tok;
      const int row_hi = P.causal ? min(pdiag + 1, kv_len) : kv_len;
      const int row_lo = P.window_left >= 0 ? max(pdiag - P.window_left, 0) : 0;
      const int b0 = (lo / POD_KBLOCK) * POD_KBLOCK;
      const int nb = (hi - b0 + POD_KBLOCK - 1) / POD_KBLOCK;
      float m_ref = NEG_INF, l = 0.f;
      for (int j = 0; j < nb; ++j) {
        const int kb = b0 + j * POD_KBLOCK;
        const int sc = s_cnt + j;
        const int b = sc & 1;
        if (!warp_wait(BAR(B_SFULL + b), (sc >> 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        float s[POD_KBLOCK];
        tmem_ld32(tmem + lane_base + L::TM_S + b * POD_KBLOCK, s);
        tmem_ld32(tmem + lane_base + L::TM_S + b * POD_KBLOCK + 32, s + 32);
        tc_fence_before();
        mbar_arrive(BAR(B_SEMPTY + b));
        const bool full = (kb >= row_lo) && (kb + POD_KBLOCK <= row_hi);
        float bmax = NEG_INF;
#pragma unroll
        for (int i = 0; i < POD_KBLOCK; ++i) {
          float x = s[i] * P.scale_log2;
          if (!full) {
            const int t = kb + i;
            if (t < row_lo || t >= row_hi) x = NEG_INF;
          }
          s[i] = x;
          bmax = fmaxf(bmax, x);
        }
        const float m_new = fmaxf(m_ref, bmax);
        const bool rescale = m_new > m_ref + 8.0f;   // also true for the first finite max
        const float m_use = rescale ? m_new : m_ref;
        const float m_sub = (m_use == NEG_INF) ? 0.f : m_use;
        float rs = 0.f;
#pragma unroll
        for (int i = 0; i < POD_KBLOCK; ++i) {
          s[i] = ex2(s[i] - m_sub);
          rs += s[i];
        }
        if (j > 0) {
          // PV of the previous block must finish before P is overwritten or O rescaled
          if (!warp_wait(BAR(B_PVDONE), pv_cnt & 1, abort_flag)) { ok = false; break; }
          ++pv_cnt;
          tc_fence_after();
          const bool need = rescale && (m_ref != NEG_INF);
          if (__any_sync(0xffffffffu, need)) {
            const float alpha = need ? ex2(m_ref - m_use) : 1.f;
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
              float o[32];
              tmem_ld32(tmem + lane_base + L::TM_O + c, o);
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] *= alpha;
              tmem_st32(tmem + lane_base + L::TM_O + c, o);
            }
            tmem_wait_st();
            l *= alpha;
          }
        }
        m_ref = m_use;
        l += rs;
        // P row -> shared memory (A operand of the PV MMA), 128B swizzle
        const uint32_t prow_addr = sbase + L::P_OFF;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t u0 = Pack<T>::two(s[8 * c + 0], s[8 * c + 1]);
          uint32_t u1 = Pack<T>::two(s[8 * c + 2], s[8 * c + 3]);
          uint32_t u2 = Pack<T>::two(s[8 * c + 4], s[8 * c + 5]);
          uint32_t u3 = Pack<T>::two(s[8 * c + 6], s[8 * c + 7]);
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(prow_addr + sw128_off(r, c)),
                       "r"(u0), "r"(u1), "r"(u2), "r"(u3)
                       : "memory");
        }
        fence_proxy_async();
        tc_fence_before();
        mbar_arrive(BAR(B_PFULL));
      }
      if (!ok) break;
      if (!warp_wait(BAR(B_PVDONE), pv_cnt & 1, abort_flag)) { ok = false; break; }
      ++pv_cnt;
      tc_fence_after();
      s_cnt += nb;
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
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    if (lane == 0) mma_commit(BAR(B_FINAL));
    __syncwarp();
    int never = 0;  // wait for the MMAs even after an abort, still bounded by the timeout
    mbar_wait(BAR(B_FINAL), 0, (volatile int*)&never);
    tc_fence_after();
    tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

// ============================================================ decode role
template <typename T, int D>
__device__ void decode_role(const PodParams& P, uint8_t* smem, int cta) {
  using L = DLayout<D>;
  constexpr bool BF16 = Pack<T>::kBF16;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int mt = warp >> 2, ks = warp & 3;
  const uint32_t sbase = smem_u32(smem);
  const int G = P.G, H = P.H;
  const T* __restrict__ qg = reinterpret_cast<const T*>(P.q_d);
  const T* __restrict__ kvg = reinterpret_cast<const T*>(P.kv_d);
  T* __restrict__ outg = reinterpret_cast<T*>(P.out_d);
  const float NEG_INF = -INFINITY;
  const int w_begin = P.cta_ptr[cta], w_end = P.cta_ptr[cta + 1];

  for (int w = w_begin; w < w_end; ++w) {
    const int32_t* rec = P.ditems + POD_REC * P.cta_list[w];
    const int req = rec[0], g = rec[1], tok0 = rec[2], ntok = rec[3], k0 = rec[4], k1 = rec[5];
    const int prow = rec[6];
    const int R = ntok * G;
    const int Mt = (R + 15) >> 4;
    const int kv_len = P.d_kv_len[req];
    const int q_base = P.d_q_indptr[req];
    const int q_len = P.d_q_indptr[req + 1] - q_base;
    const int page_base = P.d_kv_indptr[req];
    const int nst = (k1 - k0 + L::KEYS - 1) / L::KEYS;

    // Q rows (zero beyond R) go with the first stage's commit group
    for (int idx = tid; idx < POD_DECODE_ROWS * L::NCH; idx += kThreads) {
      const int r = idx / L::NCH, c = idx % L::NCH;
      const bool valid = r < R;
      const int tok = tok0 + (valid ? r / G : 0);
      const int head = g * G + (valid ? r % G : 0);
      const T* src = qg + ((size_t)(q_base + tok) * H + head) * D + c * 8;
      cp_async16(sbase + L::Q_OFF + r * L::ROWB + ((c ^ (r & 7)) << 4), src, valid ? 16u : 0u);
    }
    auto issue_stage = [&](int st) {
      const int kbase = k0 + st * L::KEYS;
      const uint32_t sb = sbase + L::STAGE_OFF + (st % L::NSTAGE) * L::STAGE_BYTES;
      constexpr int CH = L::KEYS * L::NCH;
      for (int idx = tid; idx < 2 * CH; idx += kThreads) {
        const int kv = idx / CH, rem = idx % CH;
        const int key = rem / L::NCH, c = rem % L::NCH;
        const int t = kbase + key;
        const bool valid = t < k1;
        const int tt = valid ? t : k0;
        const int pg_i = P.ps_shift >= 0 ? (tt >> P.ps_shift) : (tt / P.ps);
        const int slot = P.ps_shift >= 0 ? (tt & (P.ps - 1)) : (tt % P.ps);
        const int page = __ldg(P.d_kv_indices + page_base + pg_i);
        const T* src = kvg + ((((size_t)page * 2 + kv) * P.ps + slot) * P.Hk + g) * D + c * 8;
        cp_async16(sb + kv * L::KBYTES + key * L::ROWB + ((c ^ (key & 7)) << 4), src,
                   valid ? 16u : 0u);
      }
    };
    issue_stage(0);
    cp_async_commit();
    if (nst > 1) issue_stage(1);
    cp_async_commit();

    // rows of this thread inside its m-tile: r0 = 16 mt + lane/4, r1 = r0 + 8
    int row_lo[2], row_hi[2];
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      const int rr = mt * 16 + (lane >> 2) + 8 * h2;
      const int tok = tok0 + (rr < R ? rr / G : 0);
      const int pd = kv_len - q_len + tok;
      row_hi[h2] = P.causal ? min(pd + 1, kv_len) : kv_len;
      row_lo[h2] = P.window_left >= 0 ? max(pd - P.window_left, 0) : 0;
    }
    float m[2] = {NEG_INF, NEG_INF}, l[2] = {0.f, 0.f};
    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    const bool active = mt < Mt;

    for (int st = 0; st < nst; ++st) {
      if (st + 2 < nst) issue_stage(st + 2);
      cp_async_commit();
      cp_async_wait<2>();
      __syncthreads();
      const int kbase = k0 + st * L::KEYS + ks * 16;
      if (active && kbase < k1) {
        const uint32_t sq = sbase + L::Q_OFF;
        const uint32_t sk = sbase + L::STAGE_OFF + (st % L::NSTAGE) * L::STAGE_BYTES;
        const uint32_t sv = sk + L::KBYTES;
        float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
        const int mi = lane >> 3;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          uint32_t a[4], b[4];
          {
            const int rr = mt * 16 + (lane & 7) + ((mi & 1) << 3);
            const int c = kk * 2 + (mi >> 1);
            ldsm_x4(sq + rr * L::ROWB + ((c ^ (rr & 7)) << 4), a[0], a[1], a[2], a[3]);
          }
          {
            const int key = ks * 16 + (lane & 7) + ((mi >> 1) << 3);
            const int c = kk * 2 + (mi & 1);
            ldsm_x4(sk + key * L::ROWB + ((c ^ (key & 7)) << 4), b[0], b[1], b[2], b[3]);
          }
          mma16816<BF16>(s0, a, b[0], b[1]);
          mma16816<BF16>(s1, a, b[2], b[3]);
        }
        // scale, mask, online softmax (rows h2 = 0: c0,c1; h2 = 1: c2,c3)
        const int kq = kbase + 2 * (lane & 3);
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
            float x = *v[e] * P.scale_log2;
            if (key[e] >= k1 || key[e] < row_lo[h2] || key[e] >= row_hi[h2]) x = NEG_INF;
            *v[e] = x;
            mm = fmaxf(mm, x);
          }
          mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, 1));
          mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, 2));
          mx[h2] = mm;
        }
        uint32_t pa[4];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const float m_new = fmaxf(m[h2], mx[h2]);
          const float m_sub = (m_new == NEG_INF) ? 0.f : m_new;
          const float alpha = ex2(m[h2] - m_sub);
          m[h2] = m_new;
          float* a0 = s0 + 2 * h2;
          float* a1 = s1 + 2 * h2;
          a0[0] = ex2(a0[0] - m_sub);
          a0[1] = ex2(a0[1] - m_sub);
          a1[0] = ex2(a1[0] - m_sub);
          a1[1] = ex2(a1[1] - m_sub);
          l[h2] = l[h2] * alpha + (a0[0] + a0[1] + a1[0] + a1[1]);
#pragma unroll
          for (int i = 0; i < D / 8; ++i) {
            o[i][2 * h2] *= alpha;
            o[i][2 * h2 + 1] *= alpha;
          }
        }
        pa[0] = Pack<T>::two(s0[0], s0[1]);
        pa[1] = Pack<T>::two(s0[2], s0[3]);
        pa[2] = Pack<T>::two(s1[0], s1[1]);
        pa[3] = Pack<T>::two(s1[2], s1[3]);
#pragma unroll
        for (int j = 0; j < D / 16; ++j) {
          uint32_t b[4];
          const int key = ks * 16 + (lane & 7) + ((mi & 1) << 3);
          const int c = 2 * j + (mi >> 1);
          ldsm_x4_t(sv + key * L::ROWB + ((c ^ (key & 7)) << 4), b[0], b[1], b[2], b[3]);
          mma16816<BF16>(o[2 * j], pa, b[0], b[1]);
          mma16816<BF16>(o[2 * j + 1], pa, b[2], b[3]);
        }
      }
      __syncthreads();
    }
    cp_async_wait_all();
    __syncthreads();

    // ---- combine the 4 key slices of each m-tile through shared memory
    float* scr_o = reinterpret_cast<float*>(smem + L::SCR_O);
    float* scr_ml = reinterpret_cast<float*>(smem + L::SCR_ML);
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      l[h2] += __shfl_xor_sync(0xffffffffu, l[h2], 1);
      l[h2] += __shfl_xor_sync(0xffffffffu, l[h2], 2);
    }
    if (active) {
      float* wo = scr_o + warp * 16 * D;
#pragma unroll
      for (int i = 0; i < D / 8; ++i) {
        const int col = 8 * i + 2 * (lane & 3);
        const int rl = lane >> 2;
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
      const int tok = tok0 + rr / G;
      const int head = g * G + rr % G;
      if (prow < 0) {
        float denom = wsum;
        if (P.has_sinks) denom += ex2(P.sinks[head] * 1.4426950408889634f - Ms);
        const float inv = denom > 0.f ? 1.f / denom : 0.f;
        const size_t orow = (size_t)(q_base + tok) * H + head;
        uint2 v;
        v.x = Pack<T>::two(acc.x * inv, acc.y * inv);
        v.y = Pack<T>::two(acc.z * inv, acc.w * inv);
        *reinterpret_cast<uint2*>(outg + orow * D + c4) = v;
        if (c4 == 0 && P.lse_d) P.lse_d[orow] = wsum > 0.f ? M + log2f(wsum) : NEG_INF;
      } else {
        const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
        *reinterpret_cast<float4*>(P.part_o + (size_t)(prow + rr) * D + c4) =
            make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        if (c4 == 0) P.part_lse[prow + rr] = wsum > 0.f ? M + log2f(wsum) : NEG_INF;
      }
    }
    __syncthreads();
  }
}

// ============================================================ kernels
template <typename T, int D>
__global__ void __launch_bounds__(kThreads, POD_CTAS_PER_SM) pod_kernel(const PodParams P) {
  extern __shared__ __align__(1024) uint8_t smem[];
  // the merge kernel may start its prologue now; it waits for this grid's completion
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int cta = blockIdx.x;
  if (cta < P.n_p_ctas) {
    if ((smem_u32(smem) & 1023u) != 0u) {  // 128B-swizzle atoms need 1024-byte alignment
      if (threadIdx.x == 0) raise_status(P.status, POD_STATUS_ALIGN);
      return;
    }
    prefill_role<T, D>(P, smem, cta);
  } else {
    decode_role<T, D>(P, smem, cta);
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(256) pod_merge_kernel(const PodParams P) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int gw = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= P.n_mrows) return;
  // merge group containing merge row gw
  int lo = 0, hi = P.n_groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (P.mrow_ptr[mid] <= gw) lo = mid; else hi = mid - 1;
  }
  const int32_t* gr = P.mgroups + POD_REC * lo;
  const int half = gr[0], req = gr[1], g = gr[2], tok0 = gr[3], prow0 = gr[5], nsplit = gr[6],
            R = gr[7];
  const int r = gw - P.mrow_ptr[lo];
  const int tok = tok0 + r / P.G, head = g * P.G + r % P.G;
  float M = -INFINITY;
  for (int j = 0; j < nsplit; ++j) M = fmaxf(M, P.part_lse[prow0 + j * R + r]);
  const float Ms = (M == -INFINITY) ? 0.f : M;
  constexpr int PER = D / 32;
  float acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  float wsum = 0.f;
  for (int j = 0; j < nsplit; ++j) {
    const int pr = prow0 + j * R + r;
    const float wgt = ex2(P.part_lse[pr] - Ms);
    wsum += wgt;
    const float* src = P.part_o + (size_t)pr * D + lane * PER;
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] += wgt * src[i];
  }
  float denom = wsum;
  if (P.has_sinks) denom += ex2(P.sinks[head] * 1.4426950408889634f - Ms);
  const float inv = denom > 0.f ? 1.f / denom : 0.f;
  const int q_base = half ? P.d_q_indptr[req] : P.p_q_indptr[req];
  const size_t orow = (size_t)(q_base + tok) * P.H + head;
  T* out = reinterpret_cast<T*>(half ? P.out_d : P.out_p) + orow * D + lane * PER;
#pragma unroll
  for (int i = 0; i < PER; i += 2) {
    const uint32_t v = Pack<T>::two(acc[i] * inv, acc[i + 1] * inv);
    *reinterpret_cast<uint32_t*>(out + i) = v;
  }
  float* lse = half ? P.lse_d : P.lse_p;
  if (lane == 0 && lse) lse[orow] = wsum > 0.f ? M + log2f(wsum) : -INFINITY;
}

template <typename T, int D>
cudaError_t launch_impl(const PodParams& P, cudaStream_t stream) {
  constexpr int SMEM = smem_bytes<D>();
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(pod_kernel<T, D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    // two CTAs per SM need the largest shared-memory carveout
    e = cudaFuncSetAttribute(pod_kernel<T, D>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  if (P.grid > 0) {
    pod_kernel<T, D><<<P.grid, kThreads, SMEM, stream>>>(P);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (P.n_mrows > 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((P.n_mrows + 7) / 8));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, pod_merge_kernel<T, D>, P);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t pod_launch(const PodParams& P, int dtype, cudaStream_t stream) {
  if (P.d == 128) {
    return dtype == 1 ? launch_impl<__nv_bfloat16, 128>(P, stream)
                      : launch_impl<__half, 128>(P, stream);
  }
  return dtype == 1 ? launch_impl<__nv_bfloat16, 64>(P, stream) : launch_impl<__half, 64>(P, stream);
}

int pod_kernel_smem_bytes(int d) { return d == 128 ? smem_bytes<128>() : smem_bytes<64>(); }
