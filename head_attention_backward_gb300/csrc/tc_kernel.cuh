// Persistent KV-tile-major FMHA backward on tcgen05 tensor cores (sm_103a).
//
// Each CTA (one per SM) takes work items (segment b, kv head, KV tile of
// BN = 128 keys) from the scheduler's list, keeps that K and V tile in shared
// memory, and streams the BM = 64-row query tiles of all G query heads of the
// kv head through it.  Per (query tile, KV tile) pair it recomputes the
// scores from the stored LSE and runs the five dense products of the
// softmax-attention gradient, all with the KV tile on the 128 TMEM lanes:
//
//   S^T  = K Q^T                 (M = keys,  N = queries, K = d_qk)   SMEM x SMEM
//   dP^T = V dO^T                (M = keys,  N = queries, K = d_v)    SMEM x SMEM
//   P^T  = exp(s S^T - LSE),  dS^T = P^T o (dP^T - D)      (CUDA cores)
//   dV  += P^T dO                (M = keys,  N = d_v,     K = queries) TMEM x SMEM
//   dK  += dS^T Q                (M = keys,  N = d_qk,    K = queries) SMEM x SMEM
//   dQ^T = K^T dS^T              (M = d_qk,  N = queries, K = keys)   SMEM x SMEM
//
// P^T (TMEM) and dS^T (shared memory) are double-buffered by step parity, so
// the P/dS warps fill one buffer while the MMAs of the previous step still
// read the other.  dK and dV accumulate in TMEM across the item and are
// written once, scaled.  Each dQ^T partial (d_qk x 64 fp32) is drained from
// TMEM by four warps: stored query-major into the item's split slice of the
// dq_acc workspace (deterministic mode), or added with fp32 vector reductions
// into the single slice.  This is the persistent, deterministic split-dQ
// design of aiter PR #2216 (Motivation) re-derived for TMA + tcgen05 + TMEM.
//
// Warp roles (736 threads): warp 0 loads (TMA for Q/dO/K/V plus the LSE/D
// rows of each query tile) and fetches work items; warp 1 allocates TMEM and
// one lane issues the dV/dK/dQ^T MMAs; warp 22's lane issues the S^T/dP^T
// MMAs; warps 2-17 turn S/dP into P/dS (one key row per thread, 16 query
// columns per warp); warps 18-21 drain dQ partials and the final dK/dV.
// Every mbarrier wait is
// bounded by %globaltimer: on expiry the CTA records ATTN_ERR_TIMEOUT in the
// workspace header and all roles unwind to a clean TMEM release.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "sm100_ptx.cuh"

namespace attn {
namespace tc {

using namespace ptx;

constexpr int NUM_SOFTMAX_WARPS = 16;                  // four per scheduler
constexpr int SOFTMAX_COLS = BM * 4 / NUM_SOFTMAX_WARPS;  // query columns per softmax thread
constexpr int NUM_EPI_WARPS = 4;
constexpr int FIRST_SOFTMAX_WARP = 2;
constexpr int FIRST_EPI_WARP = FIRST_SOFTMAX_WARP + NUM_SOFTMAX_WARPS;
constexpr int SDP_ISSUER_WARP = FIRST_EPI_WARP + NUM_EPI_WARPS;   // issues the S / dP MMAs
constexpr int NUM_THREADS = 32 * (SDP_ISSUER_WARP + 1);
// ordered fold only: one more warp, whose lane 0 passes a tile's turn on once
// the drain warps' adds are issued (a 25th warp would cut the per-thread
// register budget from 80 to 72)
constexpr int TURN_WARP = SDP_ISSUER_WARP + 1;
constexpr int NUM_THREADS_FOLD = 32 * (TURN_WARP + 1);
// dQ accumulation of a kernel instantiation (each carries only its own path)
enum : int { DQ_ATOMIC = 0, DQ_FOLD = 1, DQ_SPLIT = 2 };
template <int DQM> constexpr int kernel_threads() { return DQM == DQ_FOLD ? NUM_THREADS_FOLD : NUM_THREADS; }
constexpr int NR = 4;                       // release slots between the drain and the turn thread
constexpr int NI = 2;                       // work-item ring slots
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
constexpr uint32_t SLEEP_HINT_NS = 20000;   // longest single sleep inside a wait
constexpr uint32_t TMEM_COLS = 512;

struct TmaMaps {
  CUtensorMap q, k, v, dout;
};

template <int DQK, int DV>
struct Cfg {
  // Head dims above 192 (256): dK, dV and dQ^T of a 128-key tile do not fit
  // TMEM at full width, so a KV tile is worked in NPASS passes over its query
  // tiles, pass p accumulating the 128 columns [128 p, 128 p + 128) of dK, dV
  // and dQ (S^T and dP^T are recomputed at full depth in every pass).  The
  // passes touch disjoint columns, so each is a work item of its own (the
  // work counter runs over items x passes; the item carries its pass in .w),
  // which doubles the items a GPU's SMs share.
  static constexpr int DA = DQK > 192 ? 128 : DQK;      // dK / dQ columns per pass
  static constexpr int DVA = DQK > 192 ? 128 : DV;      // dV columns per pass
  static constexpr int NPASS = DQK / DA;
  static_assert(NPASS == 1 || (DQK == DV && DQK == NPASS * DA), "multi-pass needs d_qk == d_v");
  static constexpr int NCK = DQK / 64;                  // 64-wide chunks of q/k rows
  static constexpr int NCV = DV / 64;                   // chunks of v/o rows
  static constexpr int NCA = DA / 64;                   // chunks of one pass's columns
  static constexpr int DQK_PAD = (DQK + 127) / 128 * 128;
  static constexpr int NCK_PAD = DQK_PAD / 64;          // k chunks incl. zero padding
  static constexpr int NMB = (DA + 127) / 128;          // M blocks of dQ^T per pass
  static constexpr int ST = DQK <= 128 ? 3 : DQK <= 192 ? 2 : 1;   // Q/dO pipeline stages
  static constexpr int KCH = BN * 128;                  // bytes of one 64-wide k/v chunk
  static constexpr int QCH = BM * 128;                  // bytes of one 64-wide q/dO chunk
  // TMEM column map; the two P^T buffers (bf16, two per column) are MMA A operands
  static constexpr int T_DK = 0;
  static constexpr int T_DV = DA;
  static constexpr int T_S = DA + DVA;
  static constexpr int T_DP = T_S + BM;
  static constexpr int T_DQ = T_DP + BM;
  // SEQDQ (d_qk = 192): dK and dV take 320 columns, leaving no room for two P^T
  // buffers beside S^T, dP^T and both M blocks of dQ^T.  Each thread then
  // writes its P^T (bf16 pairs) over the first half of its own S^T columns,
  // so K step ks of dV's A operand sits at T_S + 16 ks; the M blocks of dQ^T
  // take turns in one 64-column region.  dP^T of the next step is issued once
  // the P/dS warps have read dP^T, S^T of the next step once dV has read P^T.
  static constexpr bool SEQDQ = T_DQ + NMB * BM + BM > (int)TMEM_COLS;
  static constexpr int T_P = SEQDQ ? T_S : T_DQ + NMB * BM;   // P^T buffers 0 and 1 (SEQDQ: one, over S^T)
  static_assert((SEQDQ ? T_DQ + BM : T_P + BM) <= (int)TMEM_COLS, "TMEM overflow");
  static_assert(!SEQDQ || (NPASS == 1 && BM / 16 * 16 == BM), "SEQDQ: single pass");
  // shared memory map (1024-byte aligned regions)
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + NCK_PAD * KCH;
  static constexpr int OFF_Q = OFF_V + NCV * KCH;
  static constexpr int OFF_DO = OFF_Q + ST * NCK * QCH;
  static constexpr int DS_BYTES = BN * BM * 2;            // one dS^T buffer, bf16 [128 keys][64 queries]
  static constexpr int OFF_DS = OFF_DO + ST * NCV * QCH;   // two dS^T buffers (steps alternate)
  static constexpr int OFF_L = OFF_DS + 2 * DS_BYTES;      // [ST][BM] -LSE*log2(e)
  static constexpr int OFF_D = OFF_L + ST * BM * 4;        // [ST][BM] D
  static constexpr int OFF_BAR = OFF_D + ST * BM * 4;
  static constexpr int NBAR = 16 + 2 * ST + 2 * NI + 2 * NR + (NPASS > 1 ? 2 : 0);
  static constexpr int OFF_RING = OFF_BAR + NBAR * 8;
  static constexpr int OFF_MISC = OFF_RING + NI * 16;
  static constexpr int SMEM_BYTES = OFF_MISC + 64 + NR * 8 + 1024;  // + alignment slack
  static_assert(SMEM_BYTES <= 232448, "shared memory overflow");
  static_assert(OFF_BAR % 16 == 0 && OFF_RING % 16 == 0 && OFF_MISC % 16 == 0, "barrier / ring alignment");
  static constexpr uint32_t KV_BYTES = (NCK + NCV) * KCH;
  static constexpr uint32_t QDO_BYTES = (NCK + NCV) * QCH;
};

// barrier indices
// (B_PDS_FULL and B_PDS_EMPTY are pairs: one barrier per P/dS buffer)
enum {
  B_KV_FULL = 0, B_KV_EMPTY, B_SDP_FULL, B_SDP_EMPTY, B_PDS_FULL, B_PDS_EMPTY = B_PDS_FULL + 2,
  B_DQ_FULL = B_PDS_EMPTY + 2, B_DQ_EMPTY, B_DKV_FULL, B_DKV_EMPTY, B_DRAIN, B_DRAIN2,
  B_P_FREE,   // SEQDQ: dV has read the P^T written over S^T
  B_P_FULL,   // SEQDQ: P^T is in TMEM (dS^T follows with B_PDS_FULL)
  B_FIXED_END = 16
};

struct Ctx {
  uint64_t* bar;
  int* abort_flag;
  int* hdr;
};

#ifdef ATTN_WAIT_STATS
__shared__ unsigned long long g_wait_stats[48];
#endif

#ifdef ATTN_WAIT_STATS
// Optional instrumentation (off in normal builds): cycles each warp's lane 0
// spent blocked at every wait site, summed per CTA in shared memory and added
// to workspace header words [16 + 2*site] as 64-bit counters at exit.
constexpr int N_WAIT_SITES = 48;
__device__ __forceinline__ void stat_add(unsigned long long* s, int where, unsigned long long v) {
  if ((threadIdx.x & 31) == 0) atomicAdd(s + (where % N_WAIT_SITES), v);
}
#endif

// Whether a bounded wait must give up: this CTA aborted, or the wait began
// more than LIMIT ns ago (then the timeout is recorded).  Out of line: it only
// runs when a suspended try_wait returns without the phase.
template <uint64_t LIMIT>
__device__ __noinline__ bool wait_expired(const Ctx& c, uint64_t t0, int where) {
  if (*(volatile int*)c.abort_flag) return true;
  if (globaltimer() - t0 > LIMIT) {
    *(volatile int*)c.abort_flag = 1;
    atomicCAS(c.hdr + HDR_STATUS, 0, ATTN_ERR_TIMEOUT);
    atomicExch(c.hdr + HDR_DIAG, where);
    return true;
  }
  return false;
}

// Bounded mbarrier wait: one test, then suspending try_waits (the common path
// stays small at each of the many call sites: instruction-fetch stalls were
// measured to grow with the kernel's code).
template <uint64_t LIMIT = WAIT_LIMIT_NS>
__device__ __forceinline__ bool wait_bar(const Ctx& c, int idx, uint32_t parity, int where) {
  const uint32_t a = smem_u32(c.bar + idx);
  if (mbar_test_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer();
#ifdef ATTN_WAIT_STATS
  const long long c0 = clock64();
  struct Guard {
    long long c0; int where;
    __device__ ~Guard() { stat_add(g_wait_stats, where, (unsigned long long)(clock64() - c0)); }
  } guard{c0, where};
#endif
  while (!mbar_try_wait_sleep(a, parity, SLEEP_HINT_NS))
    if (wait_expired<LIMIT>(c, t0, where)) return false;
  return true;
}

// Work item and the per-item quantities every role derives identically.
struct ItemInfo {
  int b, hk, kt;
  Seg sg;
  MaskArgs m;
  int qlo, nq, nsteps, klen;
};

__device__ __forceinline__ ItemInfo item_info(const Problem& P, int4 it) {
  ItemInfo I;
  I.b = it.x; I.hk = it.y; I.kt = it.z;
  I.sg = segment(P, I.b);
  I.m = mask_args(P.mask, P.left, P.right, I.sg.lq, I.sg.lk);
  int lo, hi;
  qtile_range(I.m, I.sg.lq, I.sg.lk, I.kt, lo, hi);
  I.qlo = lo;
  I.nq = hi - lo;
  I.nsteps = I.nq * P.g;
  I.klen = min(BN, I.sg.lk - I.kt * BN);
  return I;
}

// Step s of an item -> (query head h, query tile qt).  The G query heads of
// the kv head are the inner loop and query tiles run from the last down, so
// that under the KV-tile-major item order the dQ partials of one query tile
// reach the ordered fold roughly in ascending KV-tile order.
__device__ __forceinline__ void step_coords(const Problem& P, const ItemInfo& I, int s, int& h, int& qt) {
  const int j = s / P.g;
  h = I.hk * P.g + (s - j * P.g);
  qt = I.qlo + I.nq - 1 - j;
}

// Ordered fold: poll until `rank` partials of the tile have been folded
// (bounded by %globaltimer, and given up as soon as another CTA has failed).
// The acquire load orders this warp's adds after those partials'.
template <uint64_t LIMIT = WAIT_LIMIT_NS>
__device__ __forceinline__ bool acquire_turn(const Ctx& c, const uint32_t* turn, uint32_t rank) {
  if (ld_acquire_gpu(turn) == rank) return true;
#ifdef ATTN_WAIT_STATS
  stat_add(g_wait_stats, 35, 1ull);   // turn not yet there at the second look
#endif
  const uint64_t t0 = globaltimer();
  while (ld_acquire_gpu(turn) != rank) {
    if (*(volatile int*)c.abort_flag || *(volatile int*)(c.hdr + HDR_STATUS) != 0) {
      *(volatile int*)c.abort_flag = 1;
      return false;
    }
    if (globaltimer() - t0 > LIMIT) {
      *(volatile int*)c.abort_flag = 1;
      atomicCAS(c.hdr + HDR_STATUS, 0, ATTN_ERR_TIMEOUT);
      atomicExch(c.hdr + HDR_DIAG, 33);
      return false;
    }
    __nanosleep(32);
  }
  return true;
}

// Ordered fold: (pass, query head, query tile) addresses a turn counter.
__device__ __forceinline__ bool dq_ok_turn(const Problem& P, int h, int tile) {
  return h >= 0 && h < P.hq && tile >= 0 && tile < P.ntiles;
}

template <typename T> struct IsHalf { static constexpr bool value = false; };
template <> struct IsHalf<__half> { static constexpr bool value = true; };

__device__ __forceinline__ uint32_t pack2(float a, float b, __nv_bfloat16*) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack2(float a, float b, __half*) {
  __half2 v = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// FX: the variant with attention bias, dbias and dropout (P.extras); only the
// P/dS warps differ from the plain kernel.
template <int DQK, int DV, typename T, int DQM, bool FX>
__global__ void __launch_bounds__(kernel_threads<DQM>(), 1) bwd_tc_kernel(const __grid_constant__ TmaMaps maps, const Problem P) {
  using C = Cfg<DQK, DV>;
  constexpr bool FOLD = DQM == DQ_FOLD;
  static_assert(C::NPASS == tc_passes(DQK), "turn table and workspace are sized by tc_passes()");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  int4* ring = reinterpret_cast<int4*>(smem + C::OFF_RING);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  int* abort_flag = reinterpret_cast<int*>(smem + C::OFF_MISC + 4);
  float* sL = reinterpret_cast<float*>(smem + C::OFF_L);
  float* sD = reinterpret_cast<float*>(smem + C::OFF_D);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Ctx ctx{bar, abort_flag, P.hdr};
  const int B_Q_FULL = B_FIXED_END, B_Q_EMPTY = B_FIXED_END + C::ST;
  const int B_IT_FULL = B_FIXED_END + 2 * C::ST, B_IT_EMPTY = B_IT_FULL + NI;
  // ordered fold: a partial's adds issued (drain -> turn thread) / release
  // slot free again (turn thread -> drain)
  const int B_REDS_DONE = B_IT_EMPTY + NI, B_REDS_FREE = B_REDS_DONE + NR;
  // Head dim 256 (one Q/dO stage): in pass p the column half 1 - p of Q and
  // dO feeds only S^T and dP^T, so it is loaded and released on a barrier pair
  // of its own (QA: freed by issuer A once S^T / dP^T are done, reloaded for
  // the next step during the P/dS work); the pass's own half and the row
  // statistics keep the Q_FULL / Q_EMPTY pair (freed after dV / dK).
  constexpr bool SPLITQ = C::NPASS > 1;
  const int B_QA_FULL = B_REDS_FREE + NR, B_QA_EMPTY = B_QA_FULL + 1;
  constexpr int NTHREADS = kernel_threads<DQM>();

  // zero the k padding chunks read by the dQ^T MMA of padded head dims
  if (C::NCK_PAD > C::NCK) {
    uint4* z = reinterpret_cast<uint4*>(smem + C::OFF_K + C::NCK * C::KCH);
    for (int i = threadIdx.x; i < (C::NCK_PAD - C::NCK) * C::KCH / 16; i += NTHREADS)
      z[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
#ifdef ATTN_WAIT_STATS
  if (threadIdx.x < N_WAIT_SITES) g_wait_stats[threadIdx.x] = 0;
  const long long kernel_c0 = clock64();
#endif
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar + B_KV_FULL, 1);
    mbar_init(bar + B_KV_EMPTY, 1);
    mbar_init(bar + B_SDP_FULL, 1);
    mbar_init(bar + B_SDP_EMPTY, NUM_SOFTMAX_WARPS);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar + B_PDS_FULL + b, NUM_SOFTMAX_WARPS);
      mbar_init(bar + B_PDS_EMPTY + b, 1);
    }
    mbar_init(bar + B_DQ_FULL, 1);
    mbar_init(bar + B_DQ_EMPTY, NUM_EPI_WARPS);
    mbar_init(bar + B_DKV_FULL, 1);
    mbar_init(bar + B_DKV_EMPTY, NUM_EPI_WARPS);
    mbar_init(bar + B_DRAIN, 1);
    mbar_init(bar + B_DRAIN2, 1);
    mbar_init(bar + B_P_FREE, 1);
    mbar_init(bar + B_P_FULL, NUM_SOFTMAX_WARPS);
    for (int s = 0; s < C::ST; ++s) {
      mbar_init(bar + B_Q_FULL + s, 32 + 1);   // 32 cp.async arrivals + the TMA expect_tx arrival
      mbar_init(bar + B_Q_EMPTY + s, 1);
    }
    if (SPLITQ) {
      mbar_init(bar + B_QA_FULL, 1);
      mbar_init(bar + B_QA_EMPTY, 1);
    }
    for (int s = 0; s < NI; ++s) {
      mbar_init(bar + B_IT_FULL + s, 1);
      mbar_init(bar + B_IT_EMPTY + s, 2 + NUM_SOFTMAX_WARPS + NUM_EPI_WARPS + (FOLD ? 1 : 0));
    }
    if (FOLD) {
      for (int s = 0; s < NR; ++s) {
        mbar_init(bar + B_REDS_DONE + s, NUM_EPI_WARPS);
        mbar_init(bar + B_REDS_FREE + s, 1);
      }
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const int nitems = P.hdr[HDR_NITEMS];

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&maps.q);
      tma_prefetch_desc(&maps.k);
      tma_prefetch_desc(&maps.v);
      tma_prefetch_desc(&maps.dout);
    }
    uint32_t g = 0, it = 0, n_item = 0;
    while (true) {
      int idx = 0;
      if (lane == 0) idx = atomicAdd(P.hdr + HDR_NEXT, 1);
      idx = __shfl_sync(0xffffffffu, idx, 0);
      int4 item = make_int4(-1, 0, 0, 0);
      if (idx < nitems * C::NPASS) {
        item = P.items[idx / C::NPASS];
        item.w = idx % C::NPASS;   // the pass
      }
      const int slot = n_item % NI;
      if (!wait_bar(ctx, B_IT_EMPTY + slot, ((n_item / NI) & 1) ^ 1, 1)) break;
      if (lane == 0) {
        ring[slot] = item;
        mbar_arrive(bar + B_IT_FULL + slot);
      }
      ++n_item;
      if (item.x < 0) break;
      const ItemInfo I = item_info(P, item);
      if (I.nsteps == 0) continue;
      if (!wait_bar(ctx, B_KV_EMPTY, (it & 1) ^ 1, 2)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar + B_KV_FULL, C::KV_BYTES);
        int krow = I.sg.k0 + I.kt * BN;
        if (!ATTN_INDEX_OK(P, krow >= 0 && krow < rows_k(P) && I.hk >= 0 && I.hk < P.hkv, 4)) krow = 0;
        for (int c = 0; c < C::NCK; ++c)
          tma_load_3d(smem + C::OFF_K + c * C::KCH, &maps.k, bar + B_KV_FULL, c * 64, I.hk, krow);
        for (int c = 0; c < C::NCV; ++c)
          tma_load_3d(smem + C::OFF_V + c * C::KCH, &maps.v, bar + B_KV_FULL, c * 64, I.hk, krow);
      }
      bool ok = true;
      const int nrun = I.nsteps;
      for (int s = 0; s < nrun; ++s) {
        const uint32_t gs = g + s, st = gs % C::ST;
        int h, qt;
        step_coords(P, I, s, h, qt);
        int qrow = I.sg.q0 + qt * BM;
        if (!ATTN_INDEX_OK(P, qrow >= 0 && qrow < rows_q(P) && h >= 0 && h < P.hq, 4)) qrow = 0;
        // chunks [c0, c1) of the step's Q and dO tiles onto barrier `b`
        auto load_chunks = [&](int c0, int c1, int b) {
          mbar_arrive_expect_tx(bar + b, (uint32_t)(2 * (c1 - c0)) * C::QCH);
          for (int c = c0; c < c1; ++c) {
            tma_load_3d(smem + C::OFF_Q + (st * C::NCK + c) * C::QCH, &maps.q, bar + b, c * 64, h, qrow);
            tma_load_3d(smem + C::OFF_DO + (st * C::NCV + c) * C::QCH, &maps.dout, bar + b, c * 64, h, qrow);
          }
        };
        const int pass = C::NPASS == 1 ? 0 : item.w;
        if constexpr (SPLITQ) {   // the other column half, as soon as the last S^T / dP^T are done with it
          if (!(ok = wait_bar(ctx, B_QA_EMPTY, (gs & 1) ^ 1, 7))) break;
          if (lane == 0) load_chunks((1 - pass) * C::NCA, (2 - pass) * C::NCA, B_QA_FULL);
        }
        if (!(ok = wait_bar(ctx, B_Q_EMPTY + st, ((gs / C::ST) & 1) ^ 1, 3))) break;
        auto load_tiles = [&]() {
          if (lane == 0) {
            if constexpr (SPLITQ) {
              load_chunks(pass * C::NCA, (pass + 1) * C::NCA, B_Q_FULL + st);
            } else {
              mbar_arrive_expect_tx(bar + B_Q_FULL + st, C::QDO_BYTES);
              for (int c = 0; c < C::NCK; ++c)
                tma_load_3d(smem + C::OFF_Q + (st * C::NCK + c) * C::QCH, &maps.q, bar + B_Q_FULL + st, c * 64, h,
                            qrow);
              for (int c = 0; c < C::NCV; ++c)
                tma_load_3d(smem + C::OFF_DO + (st * C::NCV + c) * C::QCH, &maps.dout, bar + B_Q_FULL + st, c * 64,
                            h, qrow);
            }
          }
        };
        // The Q / dO tiles (TMA) go first: the row statistics' per-lane copies
        // take ~1,300 cycles, which issuing the tiles after them puts on the
        // cycle a Q/dO stage goes round.  Measured faster in every mode and
        // head dim except the ordered fold at d_qk <= 128, whose cross-CTA
        // hand-offs got slower with the earlier tiles; it keeps the old order.
        constexpr bool TILES_FIRST = !FOLD || DQK > 128;
        if (TILES_FIRST) load_tiles();
        // -LSE*log2(e) and D of the tile's 64 query rows, copied asynchronously;
        // rows past the segment end read as zeros (their columns are masked)
        for (int c = lane; c < BM; c += 32) {
          const int q = qt * BM + c;
          const bool valid = q < I.sg.lq;
          long long li = valid ? lse_row(P, I.b, h, I.sg, q) : 0;
          const bool li_ok = !valid || ATTN_INDEX_OK(P, li >= 0 && li < P.n_lse, 3);
          if (!li_ok) li = 0;
          cp_async_4(sL + st * BM + c, P.nlse2 + li, valid && li_ok ? 4u : 0u);
          cp_async_4(sD + st * BM + c, P.dvec + li, valid && li_ok ? 4u : 0u);
        }
        cp_async_arrive_noinc(bar + B_Q_FULL + st);
        if (!TILES_FIRST) load_tiles();
      }
      if (!ok) break;
      g += nrun;
      ++it;
    }
  } else if (warp == 1 || warp == SDP_ISSUER_WARP) {
    // ---------------------------------------------------------- MMA issuers
    // Two single-thread issuers on different schedulers: warp SDP_ISSUER_WARP
    // issues S^T / dP^T, warp 1 (which owns the TMEM allocation) issues
    // dQ^T / dV / dK and the per-item K/V and dK/dV releases.  One thread
    // issuing every MMA, wait and commit of a step was measured as the
    // kernel's serial bottleneck.
    if (lane == 0) {
      const bool is_sdp = warp == SDP_ISSUER_WARP;
      constexpr bool F16 = IsHalf<T>::value;
      constexpr uint32_t ID_SDP = idesc_f16(128, BM, false, false, F16);
      constexpr uint32_t ID_DQ = idesc_f16(128, BM, true, true, F16);
      constexpr uint32_t ID_DV = idesc_f16(128, C::DVA, false, true, F16);
      constexpr uint32_t ID_DK = idesc_f16(128, C::DA, false, true, F16);
      // Descriptors of each operand's first 16-element K step; later steps add
      // (byte offset >> 4) to the start-address field (no carry: smem < 256 KB).
      const uint64_t dK_k = sdesc_sw128(smem_u32(smem + C::OFF_K), 16, 1024);          // K-major
      const uint64_t dV_k = sdesc_sw128(smem_u32(smem + C::OFF_V), 16, 1024);
      const uint64_t dK_mn = sdesc_sw128(smem_u32(smem + C::OFF_K), C::KCH, 1024);     // MN-major
      const uint64_t ddS_mn = sdesc_sw128(smem_u32(smem + C::OFF_DS), C::KCH, 1024);   // dQ^T B operand
      const uint64_t ddS_k = sdesc_sw128(smem_u32(smem + C::OFF_DS), 16, 1024);        // dK A operand
      const uint64_t dQ_k = sdesc_sw128(smem_u32(smem + C::OFF_Q), 16, 1024);
      const uint64_t ddO_k = sdesc_sw128(smem_u32(smem + C::OFF_DO), 16, 1024);
      const uint64_t dQ_mn = sdesc_sw128(smem_u32(smem + C::OFF_Q), C::QCH, 1024);
      const uint64_t ddO_mn = sdesc_sw128(smem_u32(smem + C::OFF_DO), C::QCH, 1024);
      uint32_t g = 0, it = 0, n_item = 0, kvp = 0;   // kvp: dK/dV accumulations handed to the drain
      bool ok = true;
      // The MMA groups are issued from straight-line code: a tcgen05.mma
      // sequence chosen per iteration by an if/else measured about twice as
      // slow per instruction on GB300, so every wait (and early exit) comes
      // before a group, never around it.
      //
      // Inputs of S^T / dP^T for global step gs are ready and their TMEM free.
      auto wait_sdp = [&](uint32_t gs) -> bool {
        return wait_bar(ctx, SPLITQ ? B_QA_FULL : B_Q_FULL + gs % C::ST, (gs / C::ST) & 1, 10) &&
               wait_bar(ctx, B_SDP_EMPTY, (gs & 1) ^ 1, 11);
      };
      // Head dim 256, pass `pass`: the K steps over the other column half of
      // Q / dO (already in) first, then, once the pass's own half is in, the
      // rest; the commit after the group frees the other half
      auto mma_sdp_split = [&](uint32_t gs, int pass) -> bool {
        const uint32_t st = gs % C::ST;
        const uint64_t q = dQ_k + ((st * C::NCK * C::QCH) >> 4), d = ddO_k + ((st * C::NCV * C::QCH) >> 4);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          if (hf == 1) {
            if (!wait_bar(ctx, B_Q_FULL + st, (gs / C::ST) & 1, 8)) return false;
            tc_fence_after();
          }
          const uint32_t cbase = (uint32_t)((hf == 0 ? 1 - pass : pass) * C::NCA);
          const uint64_t ka = dK_k + ((cbase * C::KCH) >> 4), va = dV_k + ((cbase * C::KCH) >> 4);
          const uint64_t qb = q + ((cbase * C::QCH) >> 4), db = d + ((cbase * C::QCH) >> 4);
#pragma unroll
          for (int kk = 0; kk < C::NCA * 4; ++kk) {
            const uint32_t off_a = (kk >> 2) * C::KCH + (kk & 3) * 32, off_b = (kk >> 2) * C::QCH + (kk & 3) * 32;
            umma_ss(tmem + C::T_S, ka + (off_a >> 4), qb + (off_b >> 4), ID_SDP, (hf | kk) > 0);
          }
#pragma unroll
          for (int kk = 0; kk < C::NCA * 4; ++kk) {
            const uint32_t off_a = (kk >> 2) * C::KCH + (kk & 3) * 32, off_b = (kk >> 2) * C::QCH + (kk & 3) * 32;
            umma_ss(tmem + C::T_DP, va + (off_a >> 4), db + (off_b >> 4), ID_SDP, (hf | kk) > 0);
          }
        }
        umma_commit(bar + B_SDP_FULL);
        umma_commit(bar + B_QA_EMPTY);
        return true;
      };
      // S^T = K Q^T and dP^T = V dO^T of step gs.
      auto mma_sdp = [&](uint32_t gs) -> bool {
#ifdef ATTN_WAIT_STATS
        const long long t0 = clock64();
#endif
        const uint32_t st = gs % C::ST;
        const uint64_t q = dQ_k + ((st * C::NCK * C::QCH) >> 4), d = ddO_k + ((st * C::NCV * C::QCH) >> 4);
        if constexpr (C::SEQDQ) {
          // dP^T first; S^T once dV has read the previous P^T from its columns
#pragma unroll
          for (int ks = 0; ks < DV / 16; ++ks) {
            const uint32_t off_a = (ks >> 2) * C::KCH + (ks & 3) * 32, off_b = (ks >> 2) * C::QCH + (ks & 3) * 32;
            umma_ss(tmem + C::T_DP, dV_k + (off_a >> 4), d + (off_b >> 4), ID_SDP, ks > 0);
          }
          if (!wait_bar(ctx, B_P_FREE, (gs & 1) ^ 1, 12)) return false;
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < DQK / 16; ++ks) {
            const uint32_t off_a = (ks >> 2) * C::KCH + (ks & 3) * 32, off_b = (ks >> 2) * C::QCH + (ks & 3) * 32;
            umma_ss(tmem + C::T_S, dK_k + (off_a >> 4), q + (off_b >> 4), ID_SDP, ks > 0);
          }
        } else {
#pragma unroll
        for (int ks = 0; ks < DQK / 16; ++ks) {
          const uint32_t off_a = (ks >> 2) * C::KCH + (ks & 3) * 32, off_b = (ks >> 2) * C::QCH + (ks & 3) * 32;
          umma_ss(tmem + C::T_S, dK_k + (off_a >> 4), q + (off_b >> 4), ID_SDP, ks > 0);
        }
#pragma unroll
        for (int ks = 0; ks < DV / 16; ++ks) {
          const uint32_t off_a = (ks >> 2) * C::KCH + (ks & 3) * 32, off_b = (ks >> 2) * C::QCH + (ks & 3) * 32;
          umma_ss(tmem + C::T_DP, dV_k + (off_a >> 4), d + (off_b >> 4), ID_SDP, ks > 0);
        }
        }
        umma_commit(bar + B_SDP_FULL);
#ifdef ATTN_WAIT_STATS
        stat_add(g_wait_stats, 4, (unsigned long long)(clock64() - t0));   // S/dP group issue
        stat_add(g_wait_stats, 9, 1ull);                                   // steps
#endif
        return true;
      };
      // P^T / dS^T of step gs are in their buffer (gs & 1): P^T in TMEM, dS^T
      // in shared memory.
      auto wait_pds = [&](uint32_t gs) -> bool {
        return wait_bar(ctx, B_PDS_FULL + (gs & 1), (gs >> 1) & 1, 15);
      };
      // dV += P^T dO (P^T from TMEM) and dK += dS^T Q (dS^T from shared
      // memory, K-major) of step gs, for the columns of pass `pass`; their
      // commit frees the Q/dO stage.
      auto mma_dvdk = [&](uint32_t gs, uint32_t acc_first, int pass) {
#ifdef ATTN_WAIT_STATS
        const long long t0 = clock64();
#endif
        const uint32_t st = gs % C::ST, pb = gs & 1;
        const uint64_t q = dQ_mn + (((st * C::NCK + pass * C::NCA) * C::QCH) >> 4),
                       d = ddO_mn + (((st * C::NCV + pass * C::NCA) * C::QCH) >> 4);
        const uint64_t a_ds = ddS_k + ((pb * C::DS_BYTES) >> 4);
#pragma unroll
        for (int ks = 0; ks < BM / 16; ++ks)
          umma_ts(tmem + C::T_DV, tmem + C::T_P + pb * (BM / 2) + ks * 8, d + ((ks * 2048) >> 4), ID_DV,
                  ks > 0 ? 1u : acc_first);
#pragma unroll
        for (int ks = 0; ks < BM / 16; ++ks)
          umma_ss(tmem + C::T_DK, a_ds + ((ks * 32) >> 4), q + ((ks * 2048) >> 4), ID_DK, ks > 0 ? 1u : acc_first);
        umma_commit(bar + B_Q_EMPTY + st);
#ifdef ATTN_WAIT_STATS
        stat_add(g_wait_stats, 5, (unsigned long long)(clock64() - t0));   // dV/dK group issue
#endif
      };
      // SEQDQ (single pass): dV += P^T dO with P^T over S^T, then separately
      // dK += dS^T Q, whose commit frees the Q/dO stage
      auto mma_dv = [&](uint32_t gs, uint32_t acc_first) {
        const uint64_t d = ddO_mn + (((gs % C::ST) * C::NCV * C::QCH) >> 4);
#pragma unroll
        for (int ks = 0; ks < BM / 16; ++ks)
          umma_ts(tmem + C::T_DV, tmem + C::T_S + ks * 16, d + ((ks * 2048) >> 4), ID_DV, ks > 0 ? 1u : acc_first);
      };
      auto mma_dk = [&](uint32_t gs, uint32_t acc_first) {
        const uint32_t st = gs % C::ST;
        const uint64_t q = dQ_mn + ((st * C::NCK * C::QCH) >> 4);
        const uint64_t a_ds = ddS_k + (((gs & 1) * C::DS_BYTES) >> 4);
#pragma unroll
        for (int ks = 0; ks < BM / 16; ++ks)
          umma_ss(tmem + C::T_DK, a_ds + ((ks * 32) >> 4), q + ((ks * 2048) >> 4), ID_DK, ks > 0 ? 1u : acc_first);
        umma_commit(bar + B_Q_EMPTY + st);
      };
      // The dQ^T TMEM of the previous step has been drained.
      auto wait_dq = [&](uint32_t gs) -> bool {
        return wait_bar(ctx, B_DQ_EMPTY, (gs & 1) ^ 1, 16);
      };
      // dQ^T = K^T dS^T of step gs (the rows of pass `pass`); its commit
      // also frees the P/dS buffer.
      auto mma_dq = [&](uint32_t gs, int pass) {
        const uint32_t pb = gs & 1;
        const uint64_t b_ds = ddS_mn + ((pb * C::DS_BYTES) >> 4);
#pragma unroll
        for (int mb = 0; mb < C::NMB; ++mb) {
#pragma unroll
          for (int ks = 0; ks < BN / 16; ++ks) {
            umma_ss(tmem + C::T_DQ + mb * BM, dK_mn + (((pass * C::NCA + mb * 2) * C::KCH + ks * 2048) >> 4),
                    b_ds + ((ks * 2048) >> 4), ID_DQ, ks > 0);
          }
        }
        umma_commit(bar + B_DQ_FULL);
        umma_commit(bar + B_PDS_EMPTY + pb);
      };
      // SEQDQ: M block mb of dQ^T = K^T dS^T of step gs, into the one dQ^T region
      auto mma_dq_mb = [&](uint32_t gs, int mb) {
        const uint64_t b_ds = ddS_mn + (((gs & 1) * C::DS_BYTES) >> 4);
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks)
          umma_ss(tmem + C::T_DQ, dK_mn + (((mb * 2) * C::KCH + ks * 2048) >> 4), b_ds + ((ks * 2048) >> 4), ID_DQ,
                  ks > 0);
        umma_commit(bar + B_DQ_FULL);
      };
      while (ok) {
        const int slot = n_item % NI;
        if (!wait_bar(ctx, B_IT_FULL + slot, (n_item / NI) & 1, 13)) break;
        const int4 item = ring[slot];
        mbar_arrive(bar + B_IT_EMPTY + slot);
        ++n_item;
        if (item.x < 0) break;
        const ItemInfo I = item_info(P, item);
        if (I.nsteps == 0) continue;
        const int nrun = I.nsteps;
        const uint32_t last = g + nrun - 1;
        const int pass = C::NPASS == 1 ? 0 : item.w;
        if (is_sdp) {
          if (!(ok = wait_bar(ctx, B_KV_FULL, it & 1, 14))) break;
          for (uint32_t gs = g; gs <= last; ++gs) {
            if (!(ok = wait_sdp(gs))) break;
            tc_fence_after();
            if constexpr (C::SEQDQ) {
              if (!(ok = mma_sdp(gs))) break;
            } else if constexpr (SPLITQ) {
              if (!(ok = mma_sdp_split(gs, pass))) break;
            } else {
              mma_sdp(gs);
            }
          }
        } else {
          if (!(ok = wait_bar(ctx, B_DKV_EMPTY, (kvp & 1) ^ 1, 17))) break;
          for (uint32_t gs = g; gs <= last; ++gs) {
            const bool pass_first = gs == g;
            if constexpr (C::SEQDQ) {
              // dV as soon as P^T is written (S^T of the next step waits for
              // it), dK and the dQ^T blocks once dS^T is
              if (!(ok = wait_bar(ctx, B_P_FULL, gs & 1, 24))) break;
              tc_fence_after();
              mma_dv(gs, pass_first ? 0u : 1u);
              umma_commit(bar + B_P_FREE);
              if (!(ok = wait_pds(gs))) break;
              tc_fence_after();
              mma_dk(gs, pass_first ? 0u : 1u);
#pragma unroll 1
              for (int mb = 0; mb < C::NMB; ++mb) {
                if (!(ok = wait_bar(ctx, B_DQ_EMPTY, ((gs * C::NMB + mb) & 1) ^ 1, 16))) break;
                tc_fence_after();
                mma_dq_mb(gs, mb);
              }
              if (!ok) break;
              umma_commit(bar + B_PDS_EMPTY + (gs & 1));
            } else {
            if (!(ok = wait_pds(gs))) break;
            tc_fence_after();
            mma_dvdk(gs, pass_first ? 0u : 1u, pass);
            if (!(ok = wait_dq(gs))) break;
            tc_fence_after();
            mma_dq(gs, pass);
            }
          }
          if (!ok) break;
          // the item's last dQ/dV/dK followed its last P/dS, which followed
          // every S/dP of the item: K/V and the dK/dV accumulators are done
          umma_commit(bar + B_KV_EMPTY);
          umma_commit(bar + B_DKV_FULL);
          ++kvp;
        }
        if (!ok) break;
        g += nrun;
        ++it;
      }
      // make sure no MMA of this issuer is in flight before TMEM is released
      umma_commit(bar + (is_sdp ? B_DRAIN2 : B_DRAIN));
      wait_bar(ctx, is_sdp ? B_DRAIN2 : B_DRAIN, 0, 18);
    }
  } else if (warp < FIRST_EPI_WARP) {
    // ------------------------------------------------------- softmax / dS
    const int quarter = warp & 3;
    const int grp = (warp - FIRST_SOFTMAX_WARP) >> 2;   // which SOFTMAX_COLS query columns
    const int r = quarter * 32 + lane;                   // key row = TMEM lane
    const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
    constexpr int CW = SOFTMAX_COLS;
    const int c0 = grp * CW;
    uint8_t* dsRow = smem + C::OFF_DS + r * 128;         // row r of dS^T buffer 0
    const float2 sl2 = make_float2(P.scale_log2, P.scale_log2);
    uint32_t g = 0, n_item = 0;
    while (true) {
      const int slot = n_item % NI;
      if (!wait_bar(ctx, B_IT_FULL + slot, (n_item / NI) & 1, 20)) break;
      const int4 item = ring[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar + B_IT_EMPTY + slot);
      ++n_item;
      if (item.x < 0) break;
      const ItemInfo I = item_info(P, item);
      if (I.nsteps == 0) continue;
      const int kk = I.kt * BN + r;                    // segment-local key index
      const bool key_ok = r < I.klen;
      bool ok = true;
      const int nrun = I.nsteps;
      for (int s = 0; s < nrun; ++s) {
        const uint32_t gs = g + s, st = gs % C::ST;
        int h, qt;
        step_coords(P, I, s, h, qt);
        // extras: this thread's 16 bias values (key kk, the step's query
        // columns), loaded before the S/dP wait so that it hides their latency
        uint32_t braw[FX ? CW / 2 : 1];
        if constexpr (FX) {
#pragma unroll
          for (int j = 0; j < CW / 2; ++j) braw[j] = 0u;
          if (P.bias != nullptr && key_ok) {
            const int bt = I.b + h / P.hq0, ht = h % P.hq0;   // the caller's batch entry and head
            const unsigned short* bp = static_cast<const unsigned short*>(P.bias) + bt * P.bias_sb +
                                       ht * P.bias_sh + (long long)(qt * BM + c0) * P.sk + kk;
#pragma unroll
            for (int c = 0; c < CW; ++c) {
              const uint32_t v = qt * BM + c0 + c < I.sg.lq ? __ldg(bp + (long long)c * P.sk) : 0u;
              braw[c >> 1] |= v << (16 * (c & 1));
            }
          }
        }
        if (!(ok = wait_bar(ctx, B_SDP_FULL, gs & 1, 21))) break;
        tc_fence_after();
        uint32_t sv[CW], dpv[CW];
        tmem_ld16(lane_addr + C::T_S + c0, sv);
        tmem_ld16(lane_addr + C::T_DP + c0, dpv);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar + B_SDP_EMPTY);
        if (!(ok = wait_bar(ctx, B_Q_FULL + st, (gs / C::ST) & 1, 22))) break;
        const float4* nl4 = reinterpret_cast<const float4*>(sL + st * BM + c0);
        const float4* d4 = reinterpret_cast<const float4*>(sD + st * BM + c0);
        // whole tile visible and in range: skip the per-element predicate
        const int q_first = qt * BM, q_last = qt * BM + BM - 1;
        const int k_first = I.kt * BN, k_last = I.kt * BN + BN - 1;
        const bool full = I.klen == BN && q_last < I.sg.lq &&
                          (I.m.right < 0 || k_last <= q_first + I.m.off + I.m.right) &&
                          (I.m.left < 0 || k_first >= q_last + I.m.off - I.m.left);
        uint32_t pk[CW / 2], dk[CW / 2];
        if constexpr (FX) {
          // S = scale Q K^T + bias; dropout keeps weight (q, kk) with the
          // Philox bits of its 4-row block and scales the kept ones by
          // 1 / (1 - p): P_drop feeds dV, dP o Z / (1 - p) enters dS; dbias = dS
          const int bh = I.b * P.hq + h;
          uint32_t keep = 0xFFFFu;
          if (P.drop_p > 0.f) {
            const unsigned long long seed = __ldg(P.philox_seed), offset = __ldg(P.philox_offset);
            keep = 0u;
#pragma unroll
            for (int j = 0; j < CW / 4; ++j)
              keep |= dropout_keep4(seed, offset, (uint32_t)((qt * BM + c0) / 4 + j), (uint32_t)kk, (uint32_t)bh,
                                    P.drop_thr) << (4 * j);
          }
          const float LOG2E = 1.4426950408889634f;
          T* dbias = static_cast<T*>(P.dbias);
          const long long dbase = (((long long)bh * P.sq + qt * BM + c0) * P.sk) + kk;
#pragma unroll
          for (int c = 0; c < CW; c += 2) {
            float p2[2], d2[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int cc = c + e, q = qt * BM + c0 + cc;
              const uint32_t raw = (braw[cc >> 1] >> (16 * (cc & 1))) & 0xFFFFu;
              const float bias = IsHalf<T>::value ? __half2float(__ushort_as_half((unsigned short)raw))
                                                  : __uint_as_float(raw << 16);
              const float x = fmaf(__uint_as_float(sv[cc]), P.scale_log2, fmaf(bias, LOG2E, sL[st * BM + c0 + cc]));
              const bool vis = key_ok && q < I.sg.lq && visible(I.m, q, kk);
              const float pr = vis ? fast_exp2(x) : 0.f;
              const bool kept = (keep >> cc) & 1u;
              const float f = P.drop_p > 0.f ? (kept ? P.drop_scale : 0.f) : 1.f;
              p2[e] = pr * f;
              d2[e] = pr * (__uint_as_float(dpv[cc]) * f - sD[st * BM + c0 + cc]);
              if (dbias != nullptr && key_ok && q < I.sg.lq) dbias[dbase + (long long)cc * P.sk] = TypeOps<T>::from_f(d2[e]);
            }
            pk[c >> 1] = pack2(p2[0], p2[1], (T*)nullptr);
            dk[c >> 1] = pack2(d2[0], d2[1], (T*)nullptr);
          }
        } else if constexpr (C::SEQDQ) {
          // P^T first, handed over on its own (dV and the next S^T need only
          // it), then dS^T
          float pf[CW];
#pragma unroll
          for (int c4 = 0; c4 < CW / 4; ++c4) {
            const float4 nl = nl4[c4];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const int c = 4 * c4 + 2 * hh;
              const float2 x = fma2(make_float2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sl2,
                                    hh ? make_float2(nl.z, nl.w) : make_float2(nl.x, nl.y));
              float p0 = fast_exp2(x.x), p1 = fast_exp2(x.y);
              if (!full) {
                const int q = q_first + c0 + c;
                p0 = (key_ok && q < I.sg.lq && visible(I.m, q, kk)) ? p0 : 0.f;
                p1 = (key_ok && q + 1 < I.sg.lq && visible(I.m, q + 1, kk)) ? p1 : 0.f;
              }
              pf[c] = p0;
              pf[c + 1] = p1;
              pk[c >> 1] = pack2(p0, p1, (T*)nullptr);
            }
          }
          tmem_st8(lane_addr + C::T_S + c0, pk);
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar + B_P_FULL);
#pragma unroll
          for (int c4 = 0; c4 < CW / 4; ++c4) {
            const float4 dd = d4[c4];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const int c = 4 * c4 + 2 * hh;
              const float2 ds = mul2(make_float2(pf[c], pf[c + 1]),
                                     sub2(make_float2(__uint_as_float(dpv[c]), __uint_as_float(dpv[c + 1])),
                                          hh ? make_float2(dd.z, dd.w) : make_float2(dd.x, dd.y)));
              dk[c >> 1] = pack2(ds.x, ds.y, (T*)nullptr);
            }
          }
        } else {
#pragma unroll
        for (int c4 = 0; c4 < CW / 4; ++c4) {
          const float4 nl = nl4[c4], dd = d4[c4];
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int c = 4 * c4 + 2 * hh;
            const float2 x = fma2(make_float2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sl2,
                                  hh ? make_float2(nl.z, nl.w) : make_float2(nl.x, nl.y));
            float p0 = fast_exp2(x.x), p1 = fast_exp2(x.y);
            if (!full) {
              const int q = q_first + c0 + c;
              p0 = (key_ok && q < I.sg.lq && visible(I.m, q, kk)) ? p0 : 0.f;
              p1 = (key_ok && q + 1 < I.sg.lq && visible(I.m, q + 1, kk)) ? p1 : 0.f;
            }
            const float2 p = make_float2(p0, p1);
            const float2 ds = mul2(p, sub2(make_float2(__uint_as_float(dpv[c]), __uint_as_float(dpv[c + 1])),
                                           hh ? make_float2(dd.z, dd.w) : make_float2(dd.x, dd.y)));
            pk[c >> 1] = pack2(p.x, p.y, (T*)nullptr);
            dk[c >> 1] = pack2(ds.x, ds.y, (T*)nullptr);
          }
        }
        }
        // P^T and dS^T go to buffer gs & 1; the other one may still be read
        // by the previous step's dV / dK / dQ^T MMAs
        const uint32_t pb = gs & 1;
        if constexpr (C::SEQDQ) {
          // P^T over this thread's own S^T columns (read above) needs no wait
          if constexpr (FX) {
            tmem_st8(lane_addr + C::T_S + c0, pk);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar + B_P_FULL);
          }
          if (!(ok = wait_bar(ctx, B_PDS_EMPTY + pb, ((gs >> 1) & 1) ^ 1, 23))) break;
          tc_fence_after();
        } else {
          if (!(ok = wait_bar(ctx, B_PDS_EMPTY + pb, ((gs >> 1) & 1) ^ 1, 23))) break;
          tc_fence_after();
          tmem_st8(lane_addr + C::T_P + pb * (BM / 2) + c0 / 2, pk);
        }
#pragma unroll
        for (int j = 0; j < CW / 8; ++j) {
          const int ch = grp * (CW / 8) + j;
          *reinterpret_cast<uint4*>(dsRow + pb * C::DS_BYTES + ((ch ^ (r & 7)) << 4)) =
              make_uint4(dk[4 * j], dk[4 * j + 1], dk[4 * j + 2], dk[4 * j + 3]);
        }
        if constexpr (!C::SEQDQ) tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar + B_PDS_FULL + pb);
      }
      if (!ok) break;
      g += nrun;
    }
  } else if (FOLD && warp == TURN_WARP) {
    // ------------------------------------------- ordered fold: turn thread
    // Passes on the turn of every partial whose adds all four drain warps
    // have issued: a gpu-scope fence (which waits for those adds), then the
    // tile's counter.  The drain warps acquire turns themselves; this thread
    // never waits for another CTA, so a CTA never holds back a release while
    // it waits, and every wait is for a lower KV tile, which an earlier work
    // item holds: the waits cannot form a cycle.
    if (lane == 0) {
      const uint2* rec = reinterpret_cast<const uint2*>(smem + C::OFF_MISC + 64);   // [NR] (counter, value)
      uint32_t gs = 0, n_item = 0;
      bool ok = true;
      while (ok) {
        const int slot = n_item % NI;
        if (!wait_bar(ctx, B_IT_FULL + slot, (n_item / NI) & 1, 38)) break;
        const int4 item = ring[slot];
        mbar_arrive(bar + B_IT_EMPTY + slot);
        ++n_item;
        if (item.x < 0) break;
        const ItemInfo I = item_info(P, item);
        for (int s = 0; s < I.nsteps; ++s, ++gs) {
          if (!(ok = wait_bar(ctx, B_REDS_DONE + gs % NR, (gs / NR) & 1, 40))) break;
          const uint2 r = rec[gs % NR];
#ifdef ATTN_WAIT_STATS
          const long long c0 = clock64();
#endif
          __threadfence();
          st_relaxed_gpu(P.turn + r.x, r.y);
#ifdef ATTN_WAIT_STATS
          stat_add(g_wait_stats, 34, (unsigned long long)(clock64() - c0));   // release fence
#endif
          mbar_arrive(bar + B_REDS_FREE + gs % NR);
        }
      }
    }
  } else if (warp < SDP_ISSUER_WARP) {
    // ------------------------------------------------------ dQ / dK / dV out
    const int quarter = warp & 3;
    const int L = quarter * 32 + lane;                 // TMEM lane
    const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
    T* dKg = static_cast<T*>(P.dk);
    T* dVg = static_cast<T*>(P.dv_out);
    uint32_t g = 0, kvp = 0, n_item = 0;   // kvp: dK/dV accumulations written out
    while (true) {
      const int slot = n_item % NI;
      if (!wait_bar(ctx, B_IT_FULL + slot, (n_item / NI) & 1, 30)) break;
      const int4 item = ring[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar + B_IT_EMPTY + slot);
      ++n_item;
      if (item.x < 0) break;
      const ItemInfo I = item_info(P, item);
      const int krow = I.sg.k0 + I.kt * BN + L;   // this lane's key row of dK / dV
      // element offsets of that row in dK and dV (taken here, before the step
      // loop: measured faster than at the stores)
      const long long kofs = elem_off(P.sdk_, krow, I.hk);
      const long long vofs = elem_off(P.sdv_, krow, I.hk);
      if (I.nsteps == 0) {   // no query reaches these keys: zero dK / dV (this pass's columns)
        if (L < I.klen && ATTN_INDEX_OK(P, krow >= 0 && krow < rows_k(P), 2)) {
          const int pz = C::NPASS == 1 ? 0 : item.w;
          T* dk = dKg + kofs + pz * C::DA;
          T* dv = dVg + vofs + pz * C::DVA;
          for (int e = 0; e < C::DA; ++e) dk[e] = TypeOps<T>::from_f(0.f);
          for (int e = 0; e < C::DVA; ++e) dv[e] = TypeOps<T>::from_f(0.f);
        }
        continue;
      }
      // dK (scaled) and dV of this lane's key row, the columns of pass `pass`,
      // once the issuer has committed them; then the accumulators are free
      auto write_dkdv = [&](int pass) -> bool {
        if (!wait_bar(ctx, B_DKV_FULL, kvp & 1, 32)) return false;
        tc_fence_after();
        const bool row_ok = L < I.klen && ATTN_INDEX_OK(P, krow >= 0 && krow < rows_k(P), 2);
#pragma unroll 1
        for (int ch = 0; ch < C::DA / 32; ++ch) {
          uint32_t x[32];
          tmem_ld32(lane_addr + C::T_DK + ch * 32, x);
          tmem_wait_ld();
          if (row_ok) {
            uint4* dst = reinterpret_cast<uint4*>(dKg + kofs + pass * C::DA + ch * 32);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint4 w;
              w.x = pack2(__uint_as_float(x[8 * j + 0]) * P.scale, __uint_as_float(x[8 * j + 1]) * P.scale, (T*)nullptr);
              w.y = pack2(__uint_as_float(x[8 * j + 2]) * P.scale, __uint_as_float(x[8 * j + 3]) * P.scale, (T*)nullptr);
              w.z = pack2(__uint_as_float(x[8 * j + 4]) * P.scale, __uint_as_float(x[8 * j + 5]) * P.scale, (T*)nullptr);
              w.w = pack2(__uint_as_float(x[8 * j + 6]) * P.scale, __uint_as_float(x[8 * j + 7]) * P.scale, (T*)nullptr);
              dst[j] = w;
            }
          }
        }
#pragma unroll 1
        for (int ch = 0; ch < C::DVA / 32; ++ch) {
          uint32_t x[32];
          tmem_ld32(lane_addr + C::T_DV + ch * 32, x);
          tmem_wait_ld();
          if (row_ok) {
            uint4* dst = reinterpret_cast<uint4*>(dVg + vofs + pass * C::DVA + ch * 32);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint4 w;
              w.x = pack2(__uint_as_float(x[8 * j + 0]), __uint_as_float(x[8 * j + 1]), (T*)nullptr);
              w.y = pack2(__uint_as_float(x[8 * j + 2]), __uint_as_float(x[8 * j + 3]), (T*)nullptr);
              w.z = pack2(__uint_as_float(x[8 * j + 4]), __uint_as_float(x[8 * j + 5]), (T*)nullptr);
              w.w = pack2(__uint_as_float(x[8 * j + 6]), __uint_as_float(x[8 * j + 7]), (T*)nullptr);
              dst[j] = w;
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar + B_DKV_EMPTY);
        ++kvp;
        return true;
      };
      bool ok = true;
      const int nrun = I.nsteps;
      const int pass = C::NPASS == 1 ? 0 : item.w;
      for (int s = 0; s < nrun; ++s) {
        const uint32_t gs = g + s;
        int h, qt;
        step_coords(P, I, s, h, qt);
        const int tile = qtile_index(P, I.b, qt);
        // ordered fold: this partial is number `rank` of the tile's sum; lane 0
        // of each warp reads the tile's counter before the dQ tile is ready
        uint32_t idx = 0, rank = 0, seen = ~0u;
        if (FOLD && lane == 0 && ATTN_INDEX_OK(P, dq_ok_turn(P, h, tile), 5)) {
          idx = (uint32_t)((pass * P.hq + h) * P.ntiles + tile);
          const int k0 = __ldg(P.klo + tile);
          rank = (uint32_t)(I.kt - k0);
          if (ATTN_INDEX_OK(P, k0 >= 0 && k0 <= I.kt, 6)) seen = ld_acquire_gpu(P.turn + idx);
        }
        if constexpr (!C::SEQDQ) {
          if (!(ok = wait_bar(ctx, B_DQ_FULL, gs & 1, 31))) break;
          tc_fence_after();
        }
        float* dst_tile = dq_tile(P, DQM == DQ_SPLIT ? I.kt : 0, h, tile);
        const bool dq_ok = ATTN_INDEX_OK(P, h >= 0 && h < P.hq && tile >= 0 && tile < P.ntiles &&
                                                (DQM != DQ_SPLIT || (I.kt >= 0 && I.kt < P.nsplits)), 1);
#pragma unroll 1
        for (int mb = 0; mb < C::NMB && ok; ++mb) {
          const int rows = min(128, C::DA - mb * 128);
          if constexpr (C::SEQDQ) {   // the M blocks take turns in one region
            if (!(ok = wait_bar(ctx, B_DQ_FULL, (gs * C::NMB + mb) & 1, 31))) break;
            tc_fence_after();
          }
#pragma unroll 1
          for (int hx = 0; hx < 2; ++hx) {     // query columns 0-31, then 32-63
            uint32_t v[32];
            tmem_ld32(lane_addr + C::T_DQ + (C::SEQDQ ? 0 : mb * BM) + hx * 32, v);
            tmem_wait_ld();
            if ((C::SEQDQ || mb == C::NMB - 1) && hx == 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(bar + B_DQ_EMPTY);
            }
            if (FOLD && mb == 0 && hx == 0) {
              // ordered fold: wait until the partials of the lower KV tiles are
              // in the sum (the counter read before the dQ tile was ready
              // usually shows it already)
              if (lane == 0 && seen != rank) ok = acquire_turn(ctx, P.turn + idx, rank);
              ok = __shfl_sync(0xffffffffu, ok, 0);
              if (!ok) break;
              __syncwarp();   // the other lanes' adds come after lane 0's acquire
            }
            if (L < rows && dq_ok) {
              // tile stored query-major ([BM][d_qk]): for each query the warp's
              // 32 consecutive d values fill one 128-byte line, written straight
              // from registers.  (A shared-memory staging round trip plus TMA
              // store measured ~20% slower on the whole kernel, 16-byte
              // row-segment stores slower still, d-major vector reductions
              // slower again.)
              float* dst = dst_tile + pass * C::DA + mb * 128 + L + hx * 32 * DQK;
              if constexpr (DQM == DQ_SPLIT) {   // plain store into this KV tile's slice
#pragma unroll
                for (int c = 0; c < 32; ++c) __stcg(dst + c * DQK, __uint_as_float(v[c]));
              } else {   // fp32 reductions into the zeroed slice: in arrival order
                         // (atomic) or while holding the tile's turn (ordered fold)
#pragma unroll
                for (int c = 0; c < 32; ++c) red_add_f32(dst + c * DQK, __uint_as_float(v[c]));
              }
            }
          }
        }
        if (!ok) break;
        if (FOLD) {
          // this warp's adds of the partial are issued: the turn thread passes
          // the turn on (after a gpu-scope fence) once all four warps report
          __syncwarp();
          if (lane == 0) {
            ok = wait_bar(ctx, B_REDS_FREE + gs % NR, ((gs / NR) & 1) ^ 1, 37);
            if (ok && warp == FIRST_EPI_WARP)
              reinterpret_cast<uint2*>(smem + C::OFF_MISC + 64)[gs % NR] = make_uint2(idx, rank + 1);
            if (ok) mbar_arrive(bar + B_REDS_DONE + gs % NR);
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
        }
      }
      if (!ok) break;
      g += nrun;
      if (!write_dkdv(pass)) break;
    }
  }

  tc_fence_before();
  __syncthreads();
#ifdef ATTN_WAIT_STATS
  // site 0: CTA cycles (sum over CTAs), site 19: the longest CTA
  unsigned long long* gstat = reinterpret_cast<unsigned long long*>(P.hdr + 16);
  if (threadIdx.x == 0) {
    const unsigned long long cyc = (unsigned long long)(clock64() - kernel_c0);
    g_wait_stats[0] = cyc;
    atomicMax(gstat + 19, cyc);
  }
  __syncthreads();
  if (threadIdx.x < N_WAIT_SITES && threadIdx.x != 19) atomicAdd(gstat + threadIdx.x, g_wait_stats[threadIdx.x]);
#endif
  if (warp == 1) {
    tc_fence_after();
    __syncwarp();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3-D view (dim, heads, rows) of a 16-bit tensor with element strides x;
// boxes of 64 x 1 x box_rows with 128-byte swizzle.
static bool make_map(CUtensorMap* m, const void* base, bool fp16, int dim, int heads, long long rows,
                     const Strides& x, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)dim, (cuuint64_t)heads, (cuuint64_t)(rows > 0 ? rows : 1)};
  cuuint64_t strides[2] = {(cuuint64_t)x.h * 2, (cuuint64_t)x.r * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int DQK, int DV, typename T, int DQM, bool FX>
static int launch_typed(const Problem& P, cudaStream_t st) {
  using C = Cfg<DQK, DV>;
  const bool fp16 = IsHalf<T>::value;
  TmaMaps maps;
  const long long rq = rows_q(P), rk = rows_k(P);
  if (!make_map(&maps.q, P.q, fp16, DQK, P.hq, rq, P.sq_, BM) ||
      !make_map(&maps.dout, P.dout, fp16, DV, P.hq, rq, P.sdo_, BM) ||
      !make_map(&maps.k, P.k, fp16, DQK, P.hkv, rk, P.sk_, BN) ||
      !make_map(&maps.v, P.v, fp16, DV, P.hkv, rk, P.sv_, BN))
    return ATTN_ERR_CUDA;
  auto kern = bwd_tc_kernel<DQK, DV, T, DQM, FX>;
  // at least 120 KB so that two CTAs never share an SM (each holds all 512 TMEM columns)
  const int smem = C::SMEM_BYTES > 120 * 1024 ? C::SMEM_BYTES : 120 * 1024;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return ATTN_ERR_CUDA;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int grid = sms > 0 ? sms : 1;
  const int nvirt = P.max_items * Cfg<DQK, DV>::NPASS;   // work items x passes
  if (nvirt < grid) grid = nvirt;
  if (grid <= 0) return ATTN_OK;
  // The ordered fold makes CTAs wait for one another (a partial waits for the
  // partials of lower KV tiles, which items dealt earlier hold), so that mode
  // is a cooperative launch: all CTAs are co-resident or the launch fails.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kernel_threads<DQM>());
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = DQM == DQ_FOLD ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, kern, maps, P) != cudaSuccess) return ATTN_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

template <typename T, int DQM, bool FX>
static int launch_dims(const Problem& P, cudaStream_t st) {
  if (P.dqk == 128 && P.dv == 128) return launch_typed<128, 128, T, DQM, FX>(P, st);
  if (P.dqk == 64 && P.dv == 64) return launch_typed<64, 64, T, DQM, FX>(P, st);
  if (P.dqk == 192 && P.dv == 128) return launch_typed<192, 128, T, DQM, FX>(P, st);
  if (P.dqk == 256 && P.dv == 256) return launch_typed<256, 256, T, DQM, FX>(P, st);
  return ATTN_ERR_UNSUPPORTED_HEADDIM;
}

template <typename T, bool FX>
static int launch_mode(const Problem& P, cudaStream_t st) {
  if (P.fold) return launch_dims<T, DQ_FOLD, FX>(P, st);
  return P.det ? launch_dims<T, DQ_SPLIT, FX>(P, st) : launch_dims<T, DQ_ATOMIC, FX>(P, st);
}

}  // namespace tc
}  // namespace attn
