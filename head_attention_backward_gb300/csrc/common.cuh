// Internal definitions shared by the host launcher and every kernel of the
// FMHA backward library: the problem descriptor, the workspace layout, the
// mask / tile-range arithmetic and the index helpers.  One definition of each
// layout serves the producer and the consumer of every buffer (the THD dQ bug
// of TransformerEngine PR #671, Root cause, came from two disagreeing ones).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "../../include/attn_bwd.h"

namespace attn {

// Tile shape of the backward pass: KV tiles of BN keys own a CTA; query tiles
// of BM rows stream through it.  nsplits of the deterministic dq_acc
// workspace is ceil(Sk / BN): one slice per KV tile.
constexpr int BN = 128;
constexpr int BM = 64;

// Workspace header words.
enum HeaderWord : int {
  HDR_STATUS = 0,     // attn_status_t of the last run (0 = ok)
  HDR_NITEMS = 1,     // number of work items written by the scheduler
  HDR_NEXT = 2,       // dynamic work counter of the persistent kernel
  HDR_DIAG = 3,       // diagnostic word (where a bounded wait expired)
  HDR_WORDS = 128     // words 16+: optional 64-bit wait counters of instrumented builds
};

// Element strides of a tensor seen as [rows, heads, dim] (batch entries
// folded into rows or into heads by the host); the last dimension is
// contiguous.
struct Strides {
  long long r, h;
};

struct Problem {
  // shapes
  int dtype;
  int nseg;          // B (batch) or number of segments (group)
  int hq, hkv, g;    // g = hq / hkv
  int sq, sk;        // batch: lengths; group: upper bounds
  int tq, tk;        // group: physical row totals
  int dqk, dv;
  int group;         // 1 = THD group mode
  int padded;        // group mode with a padded start array on either side
  const int* cu_q;   // logical offsets: segment lengths are their differences
  const int* cu_k;
  const int* st_q;   // physical start row of each segment (cu_q unless padded)
  const int* st_k;
  int mask, left, right;
  float scale;
  float scale_log2;  // scale * log2(e)
  int det;           // 1: bitwise-repeatable dQ (ordered fold or split slices)
  int fold;          // 1: ordered fold into one slice (see attn_det_t)
  int nsplits;       // dq_acc slices (1 unless split slices are used)
  // tensors
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const void* dout;
  const float* lse;
  void* dq;
  void* dk;
  void* dv_out;
  Strides sq_, sk_, sv_, so_, sdo_, sdq_, sdk_, sdv_;
  // workspace
  int* hdr;
  float* nlse2;      // -LSE * log2(e), -inf for rows without a visible key
  float* dvec;       // D = rowsum(dO * O)
  int4* items;       // (segment, kv head, kv tile, unused)
  int max_items;
  int* tile_off;     // group mode: first query-tile index of each segment [nseg+1]
  int ntiles;        // query tiles per (slice, head): B*ceil(Sq/BM) or an upper bound
  float* dq_acc;     // [nsplits][Hq][ntiles] query-major tiles of BM x dqk fp32 (see dq_tile)
  unsigned* turn;    // fold mode: [passes][Hq][ntiles] partials folded so far per query tile
  int* klo;          // fold mode: [ntiles] first KV tile that reaches each query tile
  long long n_lse;   // rows of the LSE layout = B*Hq*Sq or Hq*Tq
  // attention bias and dropout (the kernels' extras variant)
  int extras;        // 1: bias or dropout in use
  const void* bias;  // element (b, h, q, k) at b*bias_sb + h*bias_sh + q*sk + k
  long long bias_sb, bias_sh;
  int hq0;           // query heads of the caller's layout (the batch may be folded into the heads)
  void* dbias;       // [B, Hq, Sq, Sk] output or null
  float drop_p;      // 0 = no dropout
  float drop_scale;  // 1 / (1 - p)
  unsigned drop_thr; // keep when the Philox word >= drop_thr = floor(p * 2^32)
  const unsigned long long* philox_seed;
  const unsigned long long* philox_offset;
};

struct WsLayout {
  size_t off_hdr, off_lse2, off_dvec, off_items, off_tiles, off_turn, off_klo, off_dqacc, total;
  int max_items, nsplits, ntiles;
  bool fold;
  long long n_lse;
};

__host__ __device__ inline long long cdiv_ll(long long a, long long b) { return (a + b - 1) / b; }
__host__ __device__ inline int cdiv(int a, int b) { return (a + b - 1) / b; }

// Workspace layout: pure function of the scalar problem fields, used by both
// attn_bwd_workspace_size and attn_bwd.
// Deterministic dQ by the ordered fold: the tensor-core kernel in
// ATTN_DET_ORDERED mode (the fp32 kernel uses split slices).
inline bool det_fold(const attn_bwd_params& p) {
  return p.deterministic == ATTN_DET_ORDERED && p.dtype != ATTN_FP32;
}

// Passes per KV tile of the tensor-core kernel: head dim 256 works its dK /
// dV / dQ columns in two halves; the ordered fold keeps one turn counter per
// (pass, query head, query tile).
__host__ __device__ constexpr int tc_passes(int d_qk) { return d_qk > 192 ? 2 : 1; }

inline WsLayout ws_layout(const attn_bwd_params& p) {
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  WsLayout L{};
  const bool group = p.cu_seqlens_q != nullptr;
  L.n_lse = group ? (long long)p.nhead_q * p.total_q : (long long)p.batch * p.nhead_q * p.seqlen_q;
  L.fold = det_fold(p);
  L.nsplits = p.deterministic && !L.fold ? cdiv(p.seqlen_k > 0 ? p.seqlen_k : 1, BN) : 1;
  long long nkv_tiles;
  if (group) {
    long long a = (long long)p.total_k / BN + p.batch;
    long long b = (long long)p.batch * cdiv(p.seqlen_k > 0 ? p.seqlen_k : 1, BN);
    nkv_tiles = a < b ? a : b;
  } else {
    nkv_tiles = (long long)p.batch * cdiv(p.seqlen_k > 0 ? p.seqlen_k : 1, BN);
  }
  L.max_items = (int)(nkv_tiles * p.nhead_kv);
  if (group) {
    // sum_b ceil(Lq_b / BM) <= floor(Tq / BM) + nseg
    long long a = (long long)p.total_q / BM + p.batch;
    long long b = (long long)p.batch * cdiv(p.seqlen_q > 0 ? p.seqlen_q : 1, BM);
    L.ntiles = (int)(a < b ? a : b);
  } else {
    L.ntiles = p.batch * cdiv(p.seqlen_q, BM);
  }
  size_t o = 0;
  L.off_hdr = o;   o = up(o + HDR_WORDS * sizeof(int));
  L.off_lse2 = o;  o = up(o + (size_t)L.n_lse * sizeof(float));
  L.off_dvec = o;  o = up(o + (size_t)L.n_lse * sizeof(float));
  L.off_items = o; o = up(o + (size_t)(L.max_items > 0 ? L.max_items : 1) * sizeof(int4));
  L.off_tiles = o; o = up(o + (size_t)(p.batch + 1) * sizeof(int));
  L.off_turn = o;  o = up(o + (L.fold ? (size_t)tc_passes(p.d_qk) * p.nhead_q * L.ntiles : 1) * sizeof(unsigned));
  L.off_klo = o;   o = up(o + (L.fold ? (size_t)L.ntiles : 1) * sizeof(int));
  L.off_dqacc = o;
  o = up(o + (size_t)L.nsplits * p.nhead_q * (size_t)L.ntiles * p.d_qk * BM * sizeof(float));
  L.total = o;
  return L;
}

// ------------------------------------------------------------------ segments

struct Seg {
  int q0, lq;   // first row and length of the query segment
  int k0, lk;   // same for keys
};

// Element offset of (row, head h) of a tensor with strides x.
__host__ __device__ __forceinline__ long long elem_off(const Strides& x, long long row, int h) {
  return row * x.r + h * x.h;
}

__device__ __forceinline__ Seg segment(const Problem& P, int b) {
  Seg s;
  if (P.group) {
    s.q0 = __ldg(P.st_q + b);
    s.lq = __ldg(P.cu_q + b + 1) - __ldg(P.cu_q + b);
    s.k0 = __ldg(P.st_k + b);
    s.lk = __ldg(P.cu_k + b + 1) - __ldg(P.cu_k + b);
  } else {
    s.q0 = b * P.sq;
    s.lq = P.sq;
    s.k0 = b * P.sk;
    s.lk = P.sk;
  }
  return s;
}

// Row index of (segment b, head h, segment-local query q) in the LSE layout:
// batch [B][Hq][Sq], group [Hq][Tq] (D and the log2 LSE share it).
__device__ __forceinline__ long long lse_row(const Problem& P, int b, int h, const Seg& s, int q) {
  return P.group ? (long long)h * P.tq + s.q0 + q : ((long long)b * P.hq + h) * P.sq + q;
}

// Query-tile index of (segment b, tile qt) inside a dq_acc slice.
__device__ __forceinline__ int qtile_index(const Problem& P, int b, int qt) {
  return P.group ? __ldg(P.tile_off + b) + qt : b * cdiv(P.sq, BM) + qt;
}

// First float of the dQ tile (slice j, head h, query tile t), BM x dqk fp32,
// query-major ([BM][dqk]) in every slice.
__device__ __forceinline__ float* dq_tile(const Problem& P, int j, int h, int t) {
  return P.dq_acc + (((long long)j * P.hq + h) * P.ntiles + t) * (long long)P.dqk * BM;
}

// Global query-tile index t -> (segment b, segment-local query tile qt); false
// for indices past the last segment's tiles.  Batch mode: t = b * ceil(Sq /
// BM) + qt; group mode: the tile_off prefix written by the scheduler.
__device__ __forceinline__ bool tile_coords(const Problem& P, int t, int& b, int& qt) {
  if (P.group) {
    if (t >= __ldg(P.tile_off + P.nseg)) return false;
    int lo = 0, hi = P.nseg;                 // largest b with tile_off[b] <= t
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(P.tile_off + mid) <= t) lo = mid; else hi = mid;
    }
    b = lo;
    qt = t - __ldg(P.tile_off + b);
  } else {
    const int ntq = cdiv(P.sq, BM);
    b = t / ntq;
    qt = t - b * ntq;
  }
  return true;
}

// ---------------------------------------------------------------------- mask
// Visibility of segment-local key j to query i (same reading as the header):
// off = 0 for top-left causal, Lk - Lq for bottom-right causal and window.

struct MaskArgs {
  int off;     // diagonal offset
  int left;    // < 0: unbounded
  int right;   // < 0: unbounded
};

__host__ __device__ inline MaskArgs mask_args(int mask, int left, int right, int lq, int lk) {
  MaskArgs m;
  switch (mask) {
    case ATTN_MASK_CAUSAL_TOP_LEFT: m.off = 0; m.left = -1; m.right = 0; break;
    case ATTN_MASK_CAUSAL_BOTTOM_RIGHT: m.off = lk - lq; m.left = -1; m.right = 0; break;
    case ATTN_MASK_WINDOW: m.off = lk - lq; m.left = left; m.right = right; break;
    default: m.off = 0; m.left = -1; m.right = -1; break;
  }
  return m;
}

__host__ __device__ inline bool visible(const MaskArgs& m, int i, int j) {
  const int c = i + m.off;
  return (m.left < 0 || j >= c - m.left) && (m.right < 0 || j <= c + m.right);
}

// Range [qt_lo, qt_hi) of BM-row query tiles holding at least one query that
// sees a key of the BN-key tile kt.  Used by the main kernels (which tiles to
// visit) and by the dQ reduction (which dq_acc slices were written).
__host__ __device__ inline void qtile_range(const MaskArgs& m, int lq, int lk, int kt, int& lo, int& hi) {
  lo = 0;
  hi = 0;
  const int k_first = kt * BN;
  if (lq <= 0 || k_first >= lk) return;
  int k_last = k_first + BN - 1;
  if (k_last > lk - 1) k_last = lk - 1;
  // query i sees key j iff j - off - right <= i (right bounded) and
  // i <= j - off + left (left bounded)
  long long qlo = 0, qhi = lq - 1;
  if (m.right >= 0) {
    long long v = (long long)k_first - m.off - m.right;
    if (v > qlo) qlo = v;
  }
  if (m.left >= 0) {
    long long v = (long long)k_last - m.off + m.left;
    if (v < qhi) qhi = v;
  }
  if (qlo > qhi) return;
  lo = (int)(qlo / BM);
  hi = (int)(qhi / BM) + 1;
}

// First KV tile whose range (qtile_range) holds query tile qt, or -1 if none
// does.  Ranges only move forward with the KV tile: the tiles before the
// reached ones end at or before qt (hi <= qt), the ones after start past it or
// are empty past the last query or key.  Binary search for the first tile that
// is not "before", then check that it reaches qt.
__host__ __device__ inline int first_kv_tile(const MaskArgs& m, int lq, int lk, int qt) {
  const int nkv = (lk + BN - 1) / BN;
  auto before = [&](int kt) {
    int lo, hi;
    qtile_range(m, lq, lk, kt, lo, hi);
    if (lo < hi) return hi <= qt;
    // empty range: before the reached tiles when no query reaches this far
    // back (the left window ends before the tile), after them otherwise
    return m.left >= 0 && (long long)(kt * BN + BN - 1) - m.off + m.left < 0;
  };
  int lo = 0, hi = nkv;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (before(mid)) lo = mid + 1; else hi = mid;
  }
  if (lo >= nkv) return -1;
  int a, b;
  qtile_range(m, lq, lk, lo, a, b);
  return (a <= qt && qt < b) ? lo : -1;
}

// ------------------------------------------------------------------- types

template <typename T> struct TypeOps;
template <> struct TypeOps<__nv_bfloat16> {
  static __device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};
template <> struct TypeOps<__half> {
  static __device__ __forceinline__ float to_f(__half x) { return __half2float(x); }
  static __device__ __forceinline__ __half from_f(float x) { return __float2half_rn(x); }
};
template <> struct TypeOps<float> {
  static __device__ __forceinline__ float to_f(float x) { return x; }
  static __device__ __forceinline__ float from_f(float x) { return x; }
};

__device__ __forceinline__ void set_status(const Problem& P, int code) {
  atomicCAS(P.hdr + HDR_STATUS, 0, code);
}

// Debug builds (-DATTN_DEBUG): every computed index is checked against the
// buffer it addresses before the access.  A failing check records
// ATTN_ERR_DEVICE_FLAG and its id (HDR_DIAG = 1000 + id, first failure wins)
// in the workspace header and the access is skipped: no trap and no fault.
// Release builds compile the checks away.
#ifdef ATTN_DEBUG
static __device__ __noinline__ bool debug_index_fail(int* hdr, int id) {
  atomicCAS(hdr + HDR_STATUS, 0, ATTN_ERR_DEVICE_FLAG);
  atomicCAS(hdr + HDR_DIAG, 0, 1000 + id);
  return false;
}
#define ATTN_INDEX_OK(P, cond, id) ((cond) ? true : ::attn::debug_index_fail((P).hdr, (id)))
#else
#define ATTN_INDEX_OK(P, cond, id) true
#endif

// Rows of the q / k tensors (all batch entries, or the packed tokens).
__host__ __device__ inline long long rows_q(const Problem& P) { return P.group ? (long long)P.tq : (long long)P.nseg * P.sq; }
__host__ __device__ inline long long rows_k(const Problem& P) { return P.group ? (long long)P.tk : (long long)P.nseg * P.sk; }

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
// easy as 1, 2, 3", SC'11): ten rounds of two 32x32 -> 64-bit products with
// the published multipliers, the key bumped by the published Weyl constants
// between rounds.  c holds the counter in, the four output words out.
__device__ __forceinline__ void philox4x32_10(uint32_t (&c)[4], uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t hi0 = __umulhi(0xD2511F53u, c[0]), lo0 = 0xD2511F53u * c[0];
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c[2]), lo1 = 0xCD9E8D57u * c[2];
    const uint32_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
    c[0] = n0;
    c[1] = lo1;
    c[2] = n2;
    c[3] = lo0;
  }
}

// Dropout keep bits of query rows 4j .. 4j+3 (bit i: row 4j + i) for key
// column `col` of query head bh = b * Hq + h: counter (lo32(n), col, bh,
// hi32(n)), n = offset + j, key (lo32(seed), hi32(seed)).
__device__ __forceinline__ uint32_t dropout_keep4(unsigned long long seed, unsigned long long offset, uint32_t j,
                                                  uint32_t col, uint32_t bh, uint32_t thr) {
  const unsigned long long n = offset + j;
  uint32_t c[4] = {(uint32_t)n, col, bh, (uint32_t)(n >> 32)};
  philox4x32_10(c, (uint32_t)seed, (uint32_t)(seed >> 32));
  return (c[0] >= thr ? 1u : 0u) | (c[1] >= thr ? 2u : 0u) | (c[2] >= thr ? 4u : 0u) | (c[3] >= thr ? 8u : 0u);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------- kernel entry points

void launch_preprocess(const Problem& P, cudaStream_t st);
void launch_reduce_convert(const Problem& P, cudaStream_t st);
// A problem with no query rows or no key rows in total: resets the workspace
// header (unless keep_status) and zeroes the gradients of the other side.
void launch_empty(const Problem& P, cudaStream_t st, bool keep_status);
void launch_bwd_simt(const Problem& P, cudaStream_t st);
int launch_bwd_tc(const Problem& P, cudaStream_t st);   // returns ATTN_* status
int selftest_waits(void* scratch, size_t bytes, cudaStream_t st, int status[3]);
struct FwdLayout {
  Strides q, k, v, o;
  int hq0;                    // the caller's query heads (before a batch fold)
  long long bias_sb, bias_sh; // bias element strides of batch entry and head
};
void launch_fwd(const attn_fwd_params& p, const FwdLayout& L, cudaStream_t st);
// Forward of a problem with no key rows at all (O = 0, LSE = -inf).
void launch_fwd_no_keys(const attn_fwd_params& p, const FwdLayout& L, cudaStream_t st);

}  // namespace attn
