// Forward FMHA on tcgen05 tensor cores (sm_103a): O = softmax(s Q K^T) V and
// the natural-log LSE, for 16-bit inputs with (d_qk, d_v) in {(64, 64),
// (128, 128), (192, 128)}.  It produces the O and LSE the backward pass takes
// (the forward implied by ck_attn_fwd in TransformerEngine PR #446); fp32
// inputs and other head dims keep the CUDA-core forward in simt_kernels.cu.
//
// One CTA per (128-row query tile, query head, batch entry / segment); the
// query rows sit on the 128 TMEM lanes.  Per KV tile of 128 keys:
//
//   S  = Q K^T                 (M = queries, N = keys, K = d_qk)   SMEM x SMEM
//   P  = exp2(s log2(e) S - m) (CUDA cores, online row max m and sum l)
//   O += P V                   (M = queries, N = d_v,  K = keys)   TMEM x SMEM
//
// S is double-buffered in TMEM, so S of the next tile is computed while the
// softmax warps work on this one; K and V come in by TMA in rings of their
// own (K three tiles deep at d_qk <= 128 and freed once S is computed, V two).
// The running max is only moved (and O rescaled in TMEM) when a row's max
// grows by more than 2^8, so that P = exp2(x - m) <= 256 stays exact enough
// in 16 bits and most tiles skip the rescale.  At the end O / l goes to
// global memory and LSE = (m + log2 l) ln 2.
//
// Warp roles (352 threads): warp 0 lane 0 loads (TMA), warp 1 allocates TMEM
// and its lane 0 issues O += P V, warps 2-9 run the softmax and the epilogue
// (two warps per query row block, 64 key columns each), warp 10 lane 0 issues
// S = Q K^T.  Every wait is bounded by %globaltimer; a CTA whose wait expires
// writes NaN into its rows' LSE instead of a result.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "sm100_ptx.cuh"

namespace attn {
namespace fwdtc {

using namespace ptx;

constexpr int FM = 128;                  // query rows per CTA
constexpr int FN = 128;                  // keys per KV tile
constexpr int NUM_SM_WARPS = 8;          // softmax / epilogue warps: two per TMEM lane quarter
constexpr int SM_COLS = FN / 2;          // key columns of one softmax warp
constexpr int FIRST_SM_WARP = 2;
constexpr int S_ISSUER_WARP = FIRST_SM_WARP + NUM_SM_WARPS;   // issues S = Q K^T
constexpr int NTHREADS = 32 * (S_ISSUER_WARP + 1);
constexpr int V_STAGES = 2;              // V ring depth (K has its own ring, FCfg::KST)
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
constexpr uint32_t SLEEP_HINT_NS = 20000;
constexpr uint32_t TMEM_COLS = 512;
constexpr float RESCALE_LOG2 = 8.f;      // move the running max only past this growth

template <int DQK, int DV>
struct FCfg {
  static constexpr int NCK = DQK / 64;
  static constexpr int NCV = DV / 64;
  static constexpr int CH = 128 * 128;                    // one 64-wide chunk of 128 rows
  static constexpr int OFF_Q = 0;
  // K and V in rings of their own: a K tile is free once S = Q K^T is done,
  // so K runs KST - 1 tiles ahead; a V tile waits for its P V
  static constexpr int KST = DQK <= 128 ? 3 : 2;
  static constexpr int KSTAGE = NCK * CH;
  static constexpr int VSTAGE = NCV * CH;
  static constexpr int OFF_K = OFF_Q + NCK * CH;
  static constexpr int OFF_V = OFF_K + KST * KSTAGE;
  static constexpr int OFF_BAR = OFF_V + V_STAGES * VSTAGE;
  static constexpr int NBAR = 40;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int OFF_RED = OFF_MISC + 64;            // [3 slots][2 halves][128 rows] fp32
  static constexpr int SMEM_BYTES = OFF_RED + 3 * 2 * 128 * 4 + 1024;   // + alignment slack
  static constexpr uint32_t Q_BYTES = NCK * CH;
  static constexpr uint32_t K_BYTES = NCK * CH;
  static constexpr uint32_t V_BYTES = NCV * CH;
  // TMEM columns: two S buffers, O, two P buffers (bf16/fp16 pairs, the A
  // operand of P V; tile j uses buffer j & 1)
  static constexpr int T_S = 0;
  static constexpr int T_O = 2 * FN;
  static constexpr int T_P = T_O + 128;
  static_assert(T_P + FN <= (int)TMEM_COLS, "TMEM overflow");
  static_assert(SMEM_BYTES <= 232448, "shared memory overflow");
};

enum {
  B_Q_FULL = 0, B_K_FULL = 1, B_K_EMPTY = B_K_FULL + 3, B_V_FULL = B_K_EMPTY + 3, B_V_EMPTY = B_V_FULL + V_STAGES,
  B_S_FULL = B_V_EMPTY + V_STAGES,
  B_S_EMPTY = B_S_FULL + 2,
  // one per P buffer (tile j: j & 1).  With a single P_FULL barrier a warp
  // that has run a tile ahead would add its arrival for tile j to tile j - 1's
  // phase and release P V of j - 1 before a slower warp had written its P.
  B_P_FULL = B_S_EMPTY + 2,
  B_PV_DONE = B_P_FULL + 2,   // P V of tile j done, j & 1
  B_DRAIN = B_PV_DONE + 2, B_DRAIN2,
  // the two warps of a row block exchange row maxima per tile ([quarter][tile parity])
  // and row sums at the end ([quarter]); two lane-0 arrivals each
  B_RED, B_EPI = B_RED + 8, B_END = B_EPI + 4
};

struct Maps {
  CUtensorMap q, k, v;
};

struct Args {
  int group, hq, g, sq, sk;
  const int* cu_q;
  const int* cu_k;
  const int* st_q;
  const int* st_k;
  int mask, left, right;
  float scale_log2;
  void* o;
  Strides so;
  float* lse;
  int tq;                  // group mode: LSE row stride (rows of q)
};

struct Ctx {
  uint64_t* bar;
  int* abort_flag;
};

__device__ __noinline__ bool wait_expired(const Ctx& c, uint64_t t0) {
  if (*(volatile int*)c.abort_flag) return true;
  if (globaltimer() - t0 > WAIT_LIMIT_NS) {
    *(volatile int*)c.abort_flag = 1;
    return true;
  }
  return false;
}

__device__ __forceinline__ bool wait_bar(const Ctx& c, int idx, uint32_t parity) {
  const uint32_t a = smem_u32(c.bar + idx);
  if (mbar_test_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait_sleep(a, parity, SLEEP_HINT_NS))
    if (wait_expired(c, t0)) return false;
  return true;
}

// The same wait for all lanes of a warp, with one outcome for all of them
// (the tensor-memory loads and stores that follow are warp-collective).
__device__ __forceinline__ bool wait_bar_warp(const Ctx& c, int idx, uint32_t parity) {
  return __all_sync(0xffffffffu, wait_bar(c, idx, parity));
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

template <int DQK, int DV, typename T>
__global__ void __launch_bounds__(NTHREADS, 1) fwd_tc_kernel(const __grid_constant__ Maps maps, const Args A) {
  using C = FCfg<DQK, DV>;
  static_assert(C::KST <= 3 && B_END <= C::NBAR, "barrier slots");
  const int qt = gridDim.x - 1 - blockIdx.x;   // the longest causal tiles first
  const int h = blockIdx.y, b = blockIdx.z, hk = h / A.g;
  int q0, lq, k0, lk;
  if (A.group) {
    lq = __ldg(A.cu_q + b + 1) - __ldg(A.cu_q + b);
    lk = __ldg(A.cu_k + b + 1) - __ldg(A.cu_k + b);
    q0 = __ldg(A.st_q + b);
    k0 = __ldg(A.st_k + b);
  } else {
    q0 = b * A.sq; lq = A.sq; k0 = b * A.sk; lk = A.sk;
  }
  const int qs = qt * FM;
  if (qs >= lq) return;
  // KV tiles any row of this query tile can see
  const MaskArgs m = mask_args(A.mask, A.left, A.right, lq, lk);
  const int qe = min(qs + FM, lq) - 1;
  int klo = 0, khi = lk - 1;
  if (m.left >= 0) klo = max(klo, qs + m.off - m.left);
  if (m.right >= 0) khi = min(khi, qe + m.off + m.right);
  const int kt0 = klo / FN;
  const int nkv = (lk > 0 && khi >= klo) ? khi / FN - kt0 + 1 : 0;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  int* abort_flag = reinterpret_cast<int*>(smem + C::OFF_MISC + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Ctx ctx{bar, abort_flag};

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar + B_Q_FULL, 1);
    for (int s = 0; s < C::KST; ++s) {
      mbar_init(bar + B_K_FULL + s, 1);
      mbar_init(bar + B_K_EMPTY + s, 1);
    }
    for (int s = 0; s < V_STAGES; ++s) {
      mbar_init(bar + B_V_FULL + s, 1);
      mbar_init(bar + B_V_EMPTY + s, 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar + B_S_FULL + s, 1);
      mbar_init(bar + B_S_EMPTY + s, NUM_SM_WARPS);
    }
    mbar_init(bar + B_P_FULL, NUM_SM_WARPS);
    mbar_init(bar + B_P_FULL + 1, NUM_SM_WARPS);
    mbar_init(bar + B_PV_DONE, 1);
    mbar_init(bar + B_PV_DONE + 1, 1);
    mbar_init(bar + B_DRAIN, 1);
    mbar_init(bar + B_DRAIN2, 1);
    for (int i = B_RED; i < B_END; ++i) mbar_init(bar + i, 2);
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&maps.q);
      tma_prefetch_desc(&maps.k);
      tma_prefetch_desc(&maps.v);
      mbar_arrive_expect_tx(bar + B_Q_FULL, C::Q_BYTES);
      for (int c = 0; c < C::NCK; ++c)
        tma_load_3d(smem + C::OFF_Q + c * C::CH, &maps.q, bar + B_Q_FULL, c * 64, h, q0 + qs);
      // K tile i and V tile i - (KST - 1) in turn: K runs ahead
      constexpr int LEAD = C::KST - 1;
      int jk = 0, jv = 0;   // K / V tiles issued
      for (int i = 0; i < nkv + LEAD; ++i) {
        if (i < nkv) {
          const int s = i % C::KST;
          if (!wait_bar(ctx, B_K_EMPTY + s, ((i / C::KST) & 1) ^ 1)) break;
          mbar_arrive_expect_tx(bar + B_K_FULL + s, C::K_BYTES);
          const int krow = k0 + (kt0 + i) * FN;
          for (int c = 0; c < C::NCK; ++c)
            tma_load_3d(smem + C::OFF_K + s * C::KSTAGE + c * C::CH, &maps.k, bar + B_K_FULL + s, c * 64, hk, krow);
          ++jk;
        }
        const int v = i - LEAD;
        if (v >= 0 && v < nkv) {
          const int s = v % V_STAGES;
          if (!wait_bar(ctx, B_V_EMPTY + s, ((v / V_STAGES) & 1) ^ 1)) break;
          mbar_arrive_expect_tx(bar + B_V_FULL + s, C::V_BYTES);
          const int krow = k0 + (kt0 + v) * FN;
          for (int c = 0; c < C::NCV; ++c)
            tma_load_3d(smem + C::OFF_V + s * C::VSTAGE + c * C::CH, &maps.v, bar + B_V_FULL + s, c * 64, hk, krow);
          ++jv;
        }
      }
      // no copy may still be writing this CTA's shared memory when it exits
      wait_bar(ctx, B_Q_FULL, 0);
      for (int i = jk - 1; i >= 0 && i >= jk - C::KST; --i) wait_bar(ctx, B_K_FULL + i % C::KST, (i / C::KST) & 1);
      for (int i = jv - 1; i >= 0 && i >= jv - V_STAGES; --i) wait_bar(ctx, B_V_FULL + i % V_STAGES, (i / V_STAGES) & 1);
    }
  } else if (warp == 1 || warp == S_ISSUER_WARP) {
    // -------------------------------------------------------- MMA issuers
    // Two single-thread issuers: warp S_ISSUER_WARP issues S = Q K^T (as soon
    // as K is in and the S buffer has been read), warp 1 (which owns the TMEM
    // allocation) issues O += P V (as soon as P is written).  With one thread
    // issuing both, the next tile's S waited behind this tile's P V group.
    if (lane == 0) {
      const bool is_s = warp == S_ISSUER_WARP;
      constexpr bool F16 = IsHalf<T>::value;
      constexpr uint32_t ID_S = idesc_f16(FM, FN, false, false, F16);
      constexpr uint32_t ID_PV = idesc_f16(FM, DV, false, true, F16);
      const uint64_t dQ = sdesc_sw128(smem_u32(smem + C::OFF_Q), 16, 1024);        // K-major
      const uint64_t dK = sdesc_sw128(smem_u32(smem + C::OFF_K), 16, 1024);        // K-major, stage 0
      const uint64_t dV = sdesc_sw128(smem_u32(smem + C::OFF_V), C::CH, 1024);     // MN-major, stage 0
      bool ok = true;
      if (is_s) {
        ok = wait_bar(ctx, B_Q_FULL, 0);
        for (int j = 0; ok && j < nkv; ++j) {
          const int s = j % C::KST, sb = j & 1;
          if (!(ok = wait_bar(ctx, B_K_FULL + s, (j / C::KST) & 1))) break;
          if (!(ok = wait_bar(ctx, B_S_EMPTY + sb, ((j >> 1) & 1) ^ 1))) break;
          tc_fence_after();
          const uint64_t k = dK + ((s * C::KSTAGE) >> 4);
#pragma unroll
          for (int ks = 0; ks < DQK / 16; ++ks) {
            const uint32_t off = (ks >> 2) * C::CH + (ks & 3) * 32;
            umma_ss(tmem + C::T_S + sb * FN, dQ + (off >> 4), k + (off >> 4), ID_S, ks > 0 ? 1u : 0u);
          }
          umma_commit(bar + B_S_FULL + sb);
          umma_commit(bar + B_K_EMPTY + s);
        }
      } else {
        for (int j = 0; ok && j < nkv; ++j) {
          if (!(ok = wait_bar(ctx, B_P_FULL + (j & 1), (j >> 1) & 1))) break;
          if (!(ok = wait_bar(ctx, B_V_FULL + j % V_STAGES, (j / V_STAGES) & 1))) break;
          tc_fence_after();
          const uint64_t v = dV + (((j % V_STAGES) * C::VSTAGE) >> 4);
#pragma unroll
          for (int ks = 0; ks < FN / 16; ++ks)
            umma_ts(tmem + C::T_O, tmem + C::T_P + (j & 1) * (FN / 2) + ks * 8, v + ((ks * 2048) >> 4), ID_PV,
                    (j > 0 || ks > 0) ? 1u : 0u);
          umma_commit(bar + B_PV_DONE + (j & 1));
          umma_commit(bar + B_V_EMPTY + j % V_STAGES);
        }
      }
      // no MMA of this issuer may be in flight when TMEM is released
      umma_commit(bar + (is_s ? B_DRAIN2 : B_DRAIN));
      wait_bar(ctx, is_s ? B_DRAIN2 : B_DRAIN, 0);
    }
  } else {
    // ----------------------------------------------- softmax and epilogue
    // Warps w and w + 4 share the TMEM lanes of quarter w & 3 (query rows)
    // and take key columns [0, 64) and [64, 128) of each tile; they agree on
    // each row's max through shared memory, handing it over with an mbarrier
    // (a bounded wait, like every other wait of the kernel).
    const int quarter = warp & 3;
    const int half = (warp - FIRST_SM_WARP) >> 2;
    const int r = quarter * 32 + lane;                 // query row = TMEM lane
    const int qi = qs + r;
    const bool row_ok = qi < lq;
    const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
    float* red = reinterpret_cast<float*>(smem + C::OFF_RED);   // [slot][half][row]
    // this warp's value of row r for the partner warp: write, arrive, wait
    auto exchange = [&](float v, int slot, int b_idx, uint32_t parity, float& other) -> bool {
      red[(slot * 2 + half) * 128 + r] = v;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar + b_idx);
      if (!wait_bar_warp(ctx, b_idx, parity)) return false;
      other = red[(slot * 2 + (half ^ 1)) * 128 + r];
      return true;
    };
    constexpr int OC = DV / 2;                         // O columns of this warp
    float mx = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      const int sb = j & 1;
      if (!(ok = wait_bar_warp(ctx, B_S_FULL + sb, (j >> 1) & 1))) break;
      tc_fence_after();
      uint32_t sv[SM_COLS];
#pragma unroll
      for (int c = 0; c < SM_COLS / 32; ++c)
        tmem_ld32(lane_addr + C::T_S + sb * FN + half * SM_COLS + c * 32,
                  *reinterpret_cast<uint32_t(*)[32]>(sv + c * 32));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar + B_S_EMPTY + sb);
      // scaled scores in log2 units (masked keys -inf) and their max, with
      // independent partial maxima to keep the dependency chains short
      const int kb = (kt0 + j) * FN + half * SM_COLS;
      const bool full = kb + SM_COLS <= lk && (m.right < 0 || kb + SM_COLS - 1 <= qs + m.off + m.right) &&
                        (m.left < 0 || kb >= qe + m.off - m.left);
      // row max of the raw scores (the scale is positive), masked keys -inf
      float pm[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) pm[i] = -INFINITY;
      if (full) {   // one uniform branch per tile, not per score
#pragma unroll
        for (int c = 0; c < SM_COLS; ++c) pm[c & 7] = fmaxf(pm[c & 7], __uint_as_float(sv[c]));
      } else {
#pragma unroll
        for (int c = 0; c < SM_COLS; ++c) {
          const float x = (kb + c < lk && visible(m, qi, kb + c)) ? __uint_as_float(sv[c]) : -INFINITY;
          sv[c] = __float_as_uint(x);
          pm[c & 7] = fmaxf(pm[c & 7], x);
        }
      }
      float tmax = A.scale_log2 *
                   fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])), fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7])));
      float omax;
      if (!(ok = exchange(tmax, sb, B_RED + quarter * 2 + sb, (j >> 1) & 1, omax))) break;
      tmax = fmaxf(tmax, omax);
      // move the running max only when it grows past the threshold (both
      // warps of the pair see the same values and decide the same way)
      float alpha = 1.f;
      bool rescale = false;
      if (tmax > mx + RESCALE_LOG2) {
        alpha = fast_exp2(mx - tmax);      // 0 when mx = -inf
        rescale = j > 0;
        mx = tmax;
      }
      const float mref = mx == -INFINITY ? 0.f : mx;
      // P = exp2(s * scale log2(e) - m), two scores per packed fma
      const float2 sc2 = make_float2(A.scale_log2, A.scale_log2), nm2 = make_float2(-mref, -mref);
      const float2 one2 = make_float2(1.f, 1.f);
      float2 ps[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) ps[i] = make_float2(0.f, 0.f);
      uint32_t pk[SM_COLS / 2];
#pragma unroll
      for (int c = 0; c < SM_COLS; c += 2) {
        const float2 x = fma2(make_float2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sc2, nm2);
        const float2 p = make_float2(fast_exp2(x.x), fast_exp2(x.y));
        ps[(c >> 1) & 3] = fma2(p, one2, ps[(c >> 1) & 3]);
        pk[c >> 1] = pack2(p.x, p.y, (T*)nullptr);
      }
      l = l * alpha + (((ps[0].x + ps[0].y) + (ps[1].x + ps[1].y)) + ((ps[2].x + ps[2].y) + (ps[3].x + ps[3].y)));
      // P buffer j & 1 is free once P V of tile j - 2 is done; O may be
      // rescaled only once P V of tile j - 1 is (each buffer's barrier completes
      // once per two tiles, and tile j + 2 cannot finish before this P is written)
      if (j >= 2) {
        if (!(ok = wait_bar_warp(ctx, B_PV_DONE + (j & 1), ((j >> 1) - 1) & 1))) break;
        tc_fence_after();
      }
      const bool any_rescale = __any_sync(0xffffffffu, rescale);
      if (any_rescale) {
        if (!(ok = wait_bar_warp(ctx, B_PV_DONE + ((j - 1) & 1), ((j - 1) >> 1) & 1))) break;
        tc_fence_after();
      }
      if (any_rescale) {
#pragma unroll 1
        for (int c = 0; c < OC / 32; ++c) {
          uint32_t o[32];
          const uint32_t col = lane_addr + C::T_O + half * OC + c * 32;
          tmem_ld32(col, o);
          tmem_wait_ld();
          uint32_t lo[16], hi[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            lo[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            hi[i] = __float_as_uint(__uint_as_float(o[16 + i]) * alpha);
          }
          tmem_st16(col, lo);
          tmem_st16(col + 16, hi);
        }
      }
#pragma unroll
      for (int c = 0; c < SM_COLS / 32; ++c)
        tmem_st16(lane_addr + C::T_P + (j & 1) * (FN / 2) + half * (SM_COLS / 2) + c * 16,
                  *reinterpret_cast<const uint32_t(*)[16]>(pk + c * 16));
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar + B_P_FULL + (j & 1));
    }
    // epilogue: the row's sum over both halves, O / l (each warp its half of
    // the columns) and the LSE
    ok = __all_sync(0xffffffffu, ok);
    if (ok && nkv > 0) {
      ok = wait_bar_warp(ctx, B_PV_DONE + ((nkv - 1) & 1), ((nkv - 1) >> 1) & 1);
      tc_fence_after();
    }
    float lo_other = 0.f;
    if (ok) ok = exchange(l, 2, B_EPI + quarter, 0, lo_other);
    l += lo_other;
    const long long li = A.group ? (long long)h * A.tq + q0 + qi : ((long long)b * A.hq + h) * A.sq + qi;
    T* orow = static_cast<T*>(A.o) + elem_off(A.so, (long long)q0 + qi, h) + half * OC;
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
    for (int c = 0; c < OC / 32; ++c) {
      uint32_t o[32];
      if (ok && nkv > 0) {
        tmem_ld32(lane_addr + C::T_O + half * OC + c * 32, o);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = 0u;
      }
      if (row_ok && ok) {
        uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint4 w;
          w.x = pack2(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv, (T*)nullptr);
          w.y = pack2(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv, (T*)nullptr);
          w.z = pack2(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv, (T*)nullptr);
          w.w = pack2(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv, (T*)nullptr);
          dst[v] = w;
        }
      }
    }
    if (row_ok && half == 0)
      A.lse[li] = !ok ? __int_as_float(0x7fc00000) : l > 0.f ? (mx + log2f(l)) * 0.6931471805599453f : -INFINITY;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    __syncwarp();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side

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
// boxes of 64 x 1 x 128 rows with 128-byte swizzle.
static bool make_map(CUtensorMap* m, const void* base, bool fp16, int dim, int heads, long long rows,
                     const Strides& x) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)dim, (cuuint64_t)heads, (cuuint64_t)(rows > 0 ? rows : 1)};
  cuuint64_t strides[2] = {(cuuint64_t)x.h * 2, (cuuint64_t)x.r * 2};
  cuuint32_t box[3] = {64, 1, 128};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int DQK, int DV, typename T>
static int launch_typed(const attn_fwd_params& p, const FwdLayout& L, cudaStream_t st) {
  using C = FCfg<DQK, DV>;
  const bool group = p.cu_seqlens_q != nullptr;
  const bool fp16 = IsHalf<T>::value;
  const long long rq = group ? p.total_q : (long long)p.batch * p.seqlen_q;
  const long long rk = group ? p.total_k : (long long)p.batch * p.seqlen_k;
  Maps maps;
  if (!make_map(&maps.q, p.q, fp16, DQK, p.nhead_q, rq, L.q) || !make_map(&maps.k, p.k, fp16, DQK, p.nhead_kv, rk, L.k) ||
      !make_map(&maps.v, p.v, fp16, DV, p.nhead_kv, rk, L.v))
    return ATTN_ERR_CUDA;
  Args a;
  a.group = group ? 1 : 0;
  a.hq = p.nhead_q;
  a.g = p.nhead_q / p.nhead_kv;
  a.sq = p.seqlen_q;
  a.sk = p.seqlen_k;
  a.cu_q = p.cu_seqlens_q;
  a.cu_k = p.cu_seqlens_k;
  a.st_q = p.cu_seqlens_q_padded ? p.cu_seqlens_q_padded : p.cu_seqlens_q;
  a.st_k = p.cu_seqlens_k_padded ? p.cu_seqlens_k_padded : p.cu_seqlens_k;
  a.mask = p.mask;
  a.left = p.mask == ATTN_MASK_WINDOW ? p.window_left : -1;
  a.right = p.mask == ATTN_MASK_WINDOW ? p.window_right : -1;
  a.scale_log2 = p.softmax_scale * 1.4426950408889634f;
  a.o = p.o;
  a.so = L.o;
  a.lse = p.lse;
  a.tq = group ? p.total_q : 0;
  const int ntq = cdiv(p.seqlen_q > 0 ? p.seqlen_q : 1, FM);
  auto kern = fwd_tc_kernel<DQK, DV, T>;
  // more than half the shared memory, so that two CTAs (each holding all
  // TMEM columns) never share an SM
  const int smem = C::SMEM_BYTES > 120 * 1024 ? C::SMEM_BYTES : 120 * 1024;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return ATTN_ERR_CUDA;
  kern<<<dim3(ntq, p.nhead_q, p.batch), NTHREADS, smem, st>>>(maps, a);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

template <typename T>
static int launch_dims(const attn_fwd_params& p, const FwdLayout& L, cudaStream_t st) {
  if (p.d_qk == 128 && p.d_v == 128) return launch_typed<128, 128, T>(p, L, st);
  if (p.d_qk == 64 && p.d_v == 64) return launch_typed<64, 64, T>(p, L, st);
  if (p.d_qk == 192 && p.d_v == 128) return launch_typed<192, 128, T>(p, L, st);
  return ATTN_ERR_UNSUPPORTED_HEADDIM;
}

}  // namespace fwdtc

// Tensor-core forward for the 16-bit head-dim pairs it is built for and a
// positive softmax scale; ATTN_ERR_UNSUPPORTED_HEADDIM otherwise (the caller
// then runs the CUDA-core forward).
int launch_fwd_tc(const attn_fwd_params& p, const FwdLayout& L, cudaStream_t st) {
  // the row max is taken on the raw scores, which needs a positive scale
  if (!(p.softmax_scale > 0.f)) return ATTN_ERR_UNSUPPORTED_HEADDIM;
  if (p.dtype == ATTN_BF16) return fwdtc::launch_dims<__nv_bfloat16>(p, L, st);
  if (p.dtype == ATTN_FP16) return fwdtc::launch_dims<__half>(p, L, st);
  return ATTN_ERR_UNSUPPORTED_HEADDIM;
}

}  // namespace attn
