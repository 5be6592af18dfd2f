// Host side of the C ABI declared in include/attn_bwd.h: argument validation,
// workspace layout and the launch sequence
//   schedule -> preprocess -> main (tensor-core or fp32 SIMT) -> reduce/convert
// on the caller's stream.  Every check runs before the first CUDA call, so an
// invalid configuration is reported without touching the device (the
// "return -1" / loud-check convention of aiter PR #2216's follow-up commit
// and TransformerEngine PR #671's head-dim check).
#include <cmath>
#include <cstdio>
#include <cstdlib>

#include "common.cuh"

namespace attn {

static bool tc_headdims(int dqk, int dv) {
  return (dqk == 64 && dv == 64) || (dqk == 128 && dv == 128) || (dqk == 192 && dv == 128) ||
         (dqk == 256 && dv == 256);
}

static bool simt_headdims(int dqk, int dv) {
  return dqk >= 4 && dqk <= 64 && dv >= 1 && dv <= 64 && dqk % 4 == 0;
}

// ------------------------------------------------------------------ strides
// The kernels address every tensor as [rows, heads, dim] with a row and a
// head stride.  A batch-mode tensor fits that view when its batch entries
// follow each other along rows (batch stride = S x row stride: BSHD, packed
// QKV) -- rows are then b * S + s -- or along heads (batch stride = H x head
// stride: BHSD, SBHD) -- the problem is then run as one batch entry with
// B * Hq query and B * Hkv kv heads, which keeps the GQA grouping
// (h' / G = b * Hkv + h / G) and the [B, Hq, Sq] LSE layout.  All tensors of
// a call must fit the same way; any other layout is rejected.

struct Stride3 {
  long long b, r, h;
};

struct TensorDesc {
  const int64_t* in;   // the caller's {batch, row, head} strides
  int seqlen, heads, dim;
};

// The caller's strides, or the contiguous layout when all three are zero.
static bool resolve3(const TensorDesc& t, bool group, int batch, bool vec16, Stride3* x) {
  if (t.in[0] == 0 && t.in[1] == 0 && t.in[2] == 0) {
    x->h = t.dim;
    x->r = (long long)t.heads * t.dim;
    x->b = (long long)t.seqlen * x->r;
    return true;
  }
  x->b = t.in[0];
  x->r = t.in[1];
  x->h = t.in[2];
  const bool need_b = !group && batch > 1;
  if (x->r <= 0 || x->h <= 0 || (need_b && x->b <= 0)) return false;
  if (!need_b) x->b = (long long)t.seqlen * x->r;   // never used
  const long long lim = 1LL << 36;                    // tensor-map strides stay below 2^40 bytes
  if (x->r >= lim || x->h >= lim || x->b >= lim) return false;
  if (vec16 && (x->r % 8 || x->h % 8 || x->b % 8)) return false;
  return true;
}

// Resolves the n tensors' strides into out[] and returns 0 (rows layout),
// 1 (heads layout: fold the batch into the heads) or -1 (rejected).  A
// tensor with one row per batch entry (or one head) never uses its row (or
// head) stride, so the batch stride stands in for it; one with no rows uses
// none of its strides and constrains neither layout.
static int fold_strides(const TensorDesc* t, int n, bool group, int batch, bool vec16, Strides* out) {
  Stride3 x[8];
  bool rows = true, heads = true;
  for (int i = 0; i < n; ++i) {
    if (!resolve3(t[i], group, batch, vec16, &x[i])) return -1;
    rows &= t[i].seqlen <= 1 || x[i].b == (long long)t[i].seqlen * x[i].r;
    heads &= t[i].seqlen == 0 || t[i].heads == 1 || x[i].b == (long long)t[i].heads * x[i].h;
  }
  const int kind = (group || batch == 1 || rows) ? 0 : heads ? 1 : -1;
  for (int i = 0; i < n && kind >= 0; ++i) {
    const bool use_b = !group && batch > 1;
    out[i].r = (kind == 0 && use_b && t[i].seqlen == 1) ? x[i].b : x[i].r;
    out[i].h = (kind == 1 && t[i].heads == 1) ? x[i].b : x[i].h;
  }
  return kind;
}

// The problem the kernels run: batch folded into the heads when the layout
// asks for it, and each tensor's {row, head} strides (q, k, v, o, dout, dq,
// dk, dv).  Returns ATTN_OK or ATTN_ERR_INVALID_ARG.
static int effective_bwd(const attn_bwd_params& p, attn_bwd_params* e, Strides s[8]) {
  const bool group = p.cu_seqlens_q != nullptr;
  const TensorDesc t[8] = {{p.stride_q, p.seqlen_q, p.nhead_q, p.d_qk},   {p.stride_k, p.seqlen_k, p.nhead_kv, p.d_qk},
                           {p.stride_v, p.seqlen_k, p.nhead_kv, p.d_v},   {p.stride_o, p.seqlen_q, p.nhead_q, p.d_v},
                           {p.stride_dout, p.seqlen_q, p.nhead_q, p.d_v}, {p.stride_dq, p.seqlen_q, p.nhead_q, p.d_qk},
                           {p.stride_dk, p.seqlen_k, p.nhead_kv, p.d_qk}, {p.stride_dv, p.seqlen_k, p.nhead_kv, p.d_v}};
  const int kind = fold_strides(t, 8, group, p.batch, p.dtype != ATTN_FP32, s);
  if (kind < 0) return ATTN_ERR_INVALID_ARG;
  *e = p;
  if (kind == 1) {
    if ((long long)p.batch * p.nhead_q > (1 << 24)) return ATTN_ERR_INVALID_ARG;
    e->nhead_q = p.batch * p.nhead_q;
    e->nhead_kv = p.batch * p.nhead_kv;
    e->batch = 1;
  }
  return ATTN_OK;
}

static int effective_fwd(const attn_fwd_params& p, attn_fwd_params* e, FwdLayout* L) {
  const bool group = p.cu_seqlens_q != nullptr;
  const TensorDesc t[4] = {{p.stride_q, p.seqlen_q, p.nhead_q, p.d_qk}, {p.stride_k, p.seqlen_k, p.nhead_kv, p.d_qk},
                           {p.stride_v, p.seqlen_k, p.nhead_kv, p.d_v}, {p.stride_o, p.seqlen_q, p.nhead_q, p.d_v}};
  Strides s[4];
  const int kind = fold_strides(t, 4, group, p.batch, p.dtype != ATTN_FP32, s);
  if (kind < 0) return ATTN_ERR_INVALID_ARG;
  L->q = s[0]; L->k = s[1]; L->v = s[2]; L->o = s[3];
  L->hq0 = p.nhead_q;
  const long long mat = (long long)p.seqlen_q * p.seqlen_k;
  L->bias_sb = p.bias_type == ATTN_BIAS_BHSS ? p.nhead_q * mat : p.bias_type == ATTN_BIAS_B1SS ? mat : 0;
  L->bias_sh = p.bias_type == ATTN_BIAS_BHSS || p.bias_type == ATTN_BIAS_1HSS ? mat : 0;
  *e = p;
  if (kind == 1) {
    if ((long long)p.batch * p.nhead_q > (1 << 24)) return ATTN_ERR_INVALID_ARG;
    e->nhead_q = p.batch * p.nhead_q;
    e->nhead_kv = p.batch * p.nhead_kv;
    e->batch = 1;
  }
  return ATTN_OK;
}

template <typename Prm>
static int validate_common(const Prm* p) {
  if (!p) return ATTN_ERR_INVALID_ARG;
  if (p->dtype < ATTN_BF16 || p->dtype > ATTN_FP32) return ATTN_ERR_INVALID_ARG;
  if (p->batch < 1 || p->nhead_q < 1 || p->nhead_kv < 1) return ATTN_ERR_INVALID_ARG;
  if (p->nhead_q % p->nhead_kv != 0) return ATTN_ERR_INVALID_ARG;
  if (p->seqlen_q < 0 || p->seqlen_k < 0) return ATTN_ERR_INVALID_ARG;
  const bool gq = p->cu_seqlens_q != nullptr, gk = p->cu_seqlens_k != nullptr;
  if (gq != gk) return ATTN_ERR_INVALID_ARG;   // group mode needs both seqstart arrays
  // padded starts only refine group mode
  if (!gq && (p->cu_seqlens_q_padded || p->cu_seqlens_k_padded)) return ATTN_ERR_INVALID_ARG;
  // the seqstart arrays are read as int32 on the device
  const void* seq[] = {p->cu_seqlens_q, p->cu_seqlens_k, p->cu_seqlens_q_padded, p->cu_seqlens_k_padded};
  for (const void* x : seq)
    if ((reinterpret_cast<uintptr_t>(x) & 3u) != 0) return ATTN_ERR_INVALID_ARG;
  if (gq && (p->total_q < 0 || p->total_k < 0)) return ATTN_ERR_INVALID_ARG;
  if (p->mask < ATTN_MASK_NONE || p->mask > ATTN_MASK_WINDOW) return ATTN_ERR_INVALID_ARG;
  if (p->mask == ATTN_MASK_WINDOW && (p->window_left < -1 || p->window_right < -1))
    return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(p->softmax_scale) || p->softmax_scale == 0.f) return ATTN_ERR_INVALID_ARG;
  if (p->d_qk < 1 || p->d_v < 1) return ATTN_ERR_UNSUPPORTED_HEADDIM;
  // element counts must fit the 32-bit TMA / row coordinates
  const long long rows_q = gq ? (long long)p->total_q : (long long)p->batch * p->seqlen_q;
  const long long rows_k = gq ? (long long)p->total_k : (long long)p->batch * p->seqlen_k;
  if (rows_q > (1LL << 30) || rows_k > (1LL << 30)) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

// Attention bias and dropout fields shared by both parameter structs: the
// bias needs batch mode and a 16-bit dtype, dropout a 16-bit dtype, a
// probability in [0, 1) and both philox pointers (TE PR #446: the bias shapes
// and the philox seed / offset pointers of ck_attn_bwd).
template <typename Prm>
static int validate_extras(const Prm* p) {
  if (p->bias_type < ATTN_BIAS_NONE || p->bias_type > ATTN_BIAS_B1SS) return ATTN_ERR_INVALID_ARG;
  if (p->bias_type != ATTN_BIAS_NONE) {
    if (p->cu_seqlens_q != nullptr || p->dtype == ATTN_FP32) return ATTN_ERR_INVALID_ARG;
    if (!p->bias || (reinterpret_cast<uintptr_t>(p->bias) & 1u) != 0) return ATTN_ERR_INVALID_ARG;
  }
  if (!std::isfinite(p->dropout_p) || p->dropout_p < 0.f || p->dropout_p >= 1.f) return ATTN_ERR_INVALID_ARG;
  if (p->dropout_p > 0.f) {
    if (p->dtype == ATTN_FP32) return ATTN_ERR_INVALID_ARG;
    const void* rng[] = {p->philox_seed, p->philox_offset};
    for (const void* x : rng)
      if (!x || (reinterpret_cast<uintptr_t>(x) & 7u) != 0) return ATTN_ERR_INVALID_ARG;
  }
  return ATTN_OK;
}

static int validate_bwd(const attn_bwd_params* p) {
  int st = validate_common(p);
  if (st != ATTN_OK) return st;
  if ((st = validate_extras(p)) != ATTN_OK) return st;
  if (p->dbias && (p->bias_type == ATTN_BIAS_NONE || (reinterpret_cast<uintptr_t>(p->dbias) & 1u) != 0))
    return ATTN_ERR_INVALID_ARG;
  if (p->deterministic < ATTN_DET_ATOMIC || p->deterministic > ATTN_DET_SPLIT) return ATTN_ERR_INVALID_ARG;
  if (p->dtype == ATTN_FP32) {
    if (!simt_headdims(p->d_qk, p->d_v)) return ATTN_ERR_UNSUPPORTED_HEADDIM;
  } else if (!tc_headdims(p->d_qk, p->d_v)) {
    return ATTN_ERR_UNSUPPORTED_HEADDIM;
  }
  // 16-bit tensors feed tensor maps and 16-byte vector accesses; fp32 tensors
  // and lse are read and written one element at a time.  The tensors of a
  // side with no rows at all (no queries, or no keys) may be null.
  const bool gq = p->cu_seqlens_q != nullptr;
  const bool no_q = (gq ? (long long)p->total_q : (long long)p->batch * p->seqlen_q) == 0;
  const bool no_k = (gq ? (long long)p->total_k : (long long)p->batch * p->seqlen_k) == 0;
  const uintptr_t amask = p->dtype == ATTN_FP32 ? 3u : 15u;
  const void* ptrs[] = {p->q, p->k, p->v, p->o, p->dout, p->dq, p->dk, p->dv};
  const bool may_be_null[] = {no_q, no_k, no_k, no_q, no_q, no_q, no_k, no_k};
  for (int i = 0; i < 8; ++i)
    if ((!ptrs[i] && !may_be_null[i]) || (reinterpret_cast<uintptr_t>(ptrs[i]) & amask) != 0)
      return ATTN_ERR_INVALID_ARG;
  if ((!p->lse && !no_q) || (reinterpret_cast<uintptr_t>(p->lse) & 3u) != 0) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

static int validate_fwd(const attn_fwd_params* p) {
  int st = validate_common(p);
  if (st != ATTN_OK) return st;
  if ((st = validate_extras(p)) != ATTN_OK) return st;
  if (p->d_qk > 256 || p->d_v > 256) return ATTN_ERR_UNSUPPORTED_HEADDIM;
  // 16-bit tensors feed tensor maps and 16-byte vector stores of O (the same
  // rule as the backward's); fp32 tensors and lse are accessed one element
  // at a time.  The tensors of a side with no rows at all may be null.
  const bool gq = p->cu_seqlens_q != nullptr;
  const bool no_q = (gq ? (long long)p->total_q : (long long)p->batch * p->seqlen_q) == 0;
  const bool no_k = (gq ? (long long)p->total_k : (long long)p->batch * p->seqlen_k) == 0;
  const uintptr_t amask = p->dtype == ATTN_FP32 ? 3u : 15u;
  const void* ptrs[] = {p->q, p->k, p->v, p->o};
  const bool may_be_null[] = {no_q, no_k, no_k, no_q};
  for (int i = 0; i < 4; ++i)
    if ((!ptrs[i] && !may_be_null[i]) || (reinterpret_cast<uintptr_t>(ptrs[i]) & amask) != 0)
      return ATTN_ERR_INVALID_ARG;
  if ((!p->lse && !no_q) || (reinterpret_cast<uintptr_t>(p->lse) & 3u) != 0) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

// p: the effective problem (effective_bwd), s: its strides; hq0: the
// caller's query heads (p.nhead_q is B * hq0 when the batch is folded into
// the heads).
static Problem make_problem(const attn_bwd_params& p, const Strides s[8], void* ws, int hq0) {
  const WsLayout L = ws_layout(p);
  Problem P{};
  P.dtype = p.dtype;
  P.nseg = p.batch;
  P.hq = p.nhead_q;
  P.hkv = p.nhead_kv;
  P.g = p.nhead_q / p.nhead_kv;
  P.sq = p.seqlen_q;
  P.sk = p.seqlen_k;
  P.group = p.cu_seqlens_q != nullptr;
  P.tq = P.group ? p.total_q : p.batch * p.seqlen_q;
  P.tk = P.group ? p.total_k : p.batch * p.seqlen_k;
  P.dqk = p.d_qk;
  P.dv = p.d_v;
  P.cu_q = p.cu_seqlens_q;
  P.cu_k = p.cu_seqlens_k;
  P.st_q = p.cu_seqlens_q_padded ? p.cu_seqlens_q_padded : p.cu_seqlens_q;
  P.st_k = p.cu_seqlens_k_padded ? p.cu_seqlens_k_padded : p.cu_seqlens_k;
  P.padded = P.group && (p.cu_seqlens_q_padded || p.cu_seqlens_k_padded) ? 1 : 0;
  P.mask = p.mask;
  P.left = p.mask == ATTN_MASK_WINDOW ? p.window_left : -1;
  P.right = p.mask == ATTN_MASK_WINDOW ? p.window_right : -1;
  P.scale = p.softmax_scale;
  P.scale_log2 = p.softmax_scale * 1.4426950408889634f;
  P.det = p.deterministic != ATTN_DET_ATOMIC ? 1 : 0;
  P.fold = L.fold ? 1 : 0;
  P.nsplits = L.nsplits;
  P.q = p.q; P.k = p.k; P.v = p.v; P.o = p.o; P.dout = p.dout; P.lse = p.lse;
  P.dq = p.dq; P.dk = p.dk; P.dv_out = p.dv;
  P.sq_ = s[0]; P.sk_ = s[1]; P.sv_ = s[2]; P.so_ = s[3];
  P.sdo_ = s[4]; P.sdq_ = s[5]; P.sdk_ = s[6]; P.sdv_ = s[7];
  char* w = static_cast<char*>(ws);
  P.hdr = reinterpret_cast<int*>(w + L.off_hdr);
  P.nlse2 = reinterpret_cast<float*>(w + L.off_lse2);
  P.dvec = reinterpret_cast<float*>(w + L.off_dvec);
  P.items = reinterpret_cast<int4*>(w + L.off_items);
  P.max_items = L.max_items;
  P.tile_off = reinterpret_cast<int*>(w + L.off_tiles);
  P.ntiles = L.ntiles;
  P.dq_acc = reinterpret_cast<float*>(w + L.off_dqacc);
  P.turn = reinterpret_cast<unsigned*>(w + L.off_turn);
  P.klo = reinterpret_cast<int*>(w + L.off_klo);
  P.n_lse = L.n_lse;
  P.hq0 = hq0;
  P.extras = p.bias_type != ATTN_BIAS_NONE || p.dropout_p > 0.f;
  if (p.bias_type != ATTN_BIAS_NONE) {
    const long long mat = (long long)p.seqlen_q * p.seqlen_k;   // one [Sq, Sk] matrix
    P.bias = p.bias;
    P.bias_sb = p.bias_type == ATTN_BIAS_BHSS ? hq0 * mat : p.bias_type == ATTN_BIAS_B1SS ? mat : 0;
    P.bias_sh = p.bias_type == ATTN_BIAS_BHSS || p.bias_type == ATTN_BIAS_1HSS ? mat : 0;
    P.dbias = p.dbias;
  }
  if (p.dropout_p > 0.f) {
    P.drop_p = p.dropout_p;
    P.drop_scale = 1.f / (1.f - p.dropout_p);
    const double t = std::floor((double)p.dropout_p * 4294967296.0);
    P.drop_thr = t >= 4294967295.0 ? 4294967295u : (unsigned)t;
    P.philox_seed = reinterpret_cast<const unsigned long long*>(p.philox_seed);
    P.philox_offset = reinterpret_cast<const unsigned long long*>(p.philox_offset);
  }
  return P;
}

static bool log_enabled() {
  const char* e = std::getenv("ATTN_BWD_LOG");
  return e && e[0] == '1';
}

static void log_config(const attn_bwd_params& p, const WsLayout& L) {
  std::fprintf(stderr,
               "[attn_bwd] dtype=%d mode=%s batch=%d hq=%d hkv=%d sq=%d sk=%d tq=%d tk=%d d_qk=%d d_v=%d "
               "mask=%d window=(%d,%d) scale=%g det=%d nsplits=%d items<=%d workspace=%zu\n",
               p.dtype,
               p.cu_seqlens_q ? (p.cu_seqlens_q_padded || p.cu_seqlens_k_padded ? "group-padded" : "group")
                              : "batch", p.batch, p.nhead_q, p.nhead_kv, p.seqlen_q,
               p.seqlen_k, p.total_q, p.total_k, p.d_qk, p.d_v, p.mask, p.window_left, p.window_right,
               p.softmax_scale, p.deterministic, L.nsplits, L.max_items, L.total);
}

// Tensor-core forward (fwd_tc.cu); ATTN_ERR_UNSUPPORTED_HEADDIM for the
// dtypes and head dims it is not built for.
int launch_fwd_tc(const attn_fwd_params& p, const FwdLayout& L, cudaStream_t st);

// Schedule and preprocess launches of one call, or of one part of a call
// split into parts (attn_bwd_host: parts after the first keep the status the
// earlier parts left).
void launch_schedule_preprocess(const Problem& P, cudaStream_t st, bool keep_status);

// The validated problem the kernels of one call (or of one part of a call) run.
static int prepare(const attn_bwd_params* p, void* ws, size_t ws_bytes, Problem* P) {
  int st = validate_bwd(p);
  if (st != ATTN_OK) return st;
  attn_bwd_params e;
  Strides sx[8];
  if ((st = effective_bwd(*p, &e, sx)) != ATTN_OK) return st;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return ATTN_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(e);
  if (ws_bytes < L.total) return ATTN_ERR_WORKSPACE_TOO_SMALL;
  if (log_enabled()) log_config(e, L);
  *P = make_problem(e, sx, ws, p->nhead_q);
  return ATTN_OK;
}

// The main kernel: tensor cores for 16-bit inputs, CUDA cores for fp32.  It
// leaves dK and dV final; dQ is final after the reduce/convert kernel.
static int launch_main(const Problem& P, cudaStream_t s) {
  if (P.dtype == ATTN_FP32) {
    launch_bwd_simt(P, s);
    return ATTN_OK;
  }
  return launch_bwd_tc(P, s);
}

// No query rows or no key rows in total: the gradients of the other side are
// zero and no attention kernel runs.
static bool empty_problem(const Problem& P) { return rows_q(P) == 0 || rows_k(P) == 0; }

static int run(const attn_bwd_params* p, void* ws, size_t ws_bytes, cudaStream_t s,
               cudaEvent_t* ev /* 4 events or null */, bool keep_status = false) {
  Problem P;
  int st = prepare(p, ws, ws_bytes, &P);
  if (st != ATTN_OK) return st;
  if (ev) cudaEventRecord(ev[0], s);
  if (empty_problem(P)) {
    launch_empty(P, s, keep_status);
    for (int i = 1; ev && i < 4; ++i) cudaEventRecord(ev[i], s);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
  }
  launch_schedule_preprocess(P, s, keep_status);
  if (ev) cudaEventRecord(ev[1], s);
  if ((st = launch_main(P, s)) != ATTN_OK) return st;
  if (ev) cudaEventRecord(ev[2], s);
  launch_reduce_convert(P, s);
  if (ev) cudaEventRecord(ev[3], s);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

static bool all_zero(const int64_t x[3]) { return x[0] == 0 && x[1] == 0 && x[2] == 0; }

static size_t dtype_bytes(int dtype) { return dtype == ATTN_FP32 ? 4 : 2; }

// One tensor of attn_bwd_host: rows per batch entry (all rows in group mode),
// heads, head dim, element bytes.
struct HostTensor {
  long long rows;
  int heads, dim;
  size_t es;
};

// Copies rows [b0 * rows, b1 * rows) x heads [x0, x1) of a contiguous tensor
// between host and device: one plain copy when the heads are all of them,
// else a 2-D copy (one row's head slice per line).
static bool copy_part(const HostTensor& t, void* dst, const void* src, int b0, int b1, int x0, int x1,
                      cudaMemcpyKind kind, cudaStream_t st) {
  const size_t row = (size_t)t.heads * t.dim * t.es;
  const size_t off = (size_t)b0 * t.rows * row + (size_t)x0 * t.dim * t.es;
  char* d = static_cast<char*>(dst) + off;
  const char* s = static_cast<const char*>(src) + off;
  const size_t nrows = (size_t)(b1 - b0) * t.rows;
  if (nrows == 0) return true;
  if (x0 == 0 && x1 == t.heads) return cudaMemcpyAsync(d, s, nrows * row, kind, st) == cudaSuccess;
  return cudaMemcpy2DAsync(d, row, s, row, (size_t)(x1 - x0) * t.dim * t.es, nrows, kind, st) == cudaSuccess;
}

// Chunked host <-> device pipeline of attn_bwd_host.  A chunk is a run of
// batch entries or, once there are more chunks than entries, one entry (or
// the whole packed tensor in group mode) and a run of kv heads with their
// query heads; either way its LSE rows are one contiguous block.  Its inputs
// go up on `in`, its backward runs on `s` (on strided views of the staging
// buffers), its gradients come down on `out`; events order the three, so the
// copies of one chunk overlap the compute of its neighbours.
static int run_host(const attn_bwd_params* p, const attn_host_tensors* h, void* ws, size_t ws_bytes, cudaStream_t s,
                    cudaStream_t in, cudaStream_t out, int chunks) {
  int st = validate_bwd(p);
  if (st != ATTN_OK) return st;
  if (!h) return ATTN_ERR_INVALID_ARG;
  {  // as on the device side, a side with no rows at all may have null tensors
    const bool gq = p->cu_seqlens_q != nullptr;
    const bool no_q = (gq ? (long long)p->total_q : (long long)p->batch * p->seqlen_q) == 0;
    const bool no_k = (gq ? (long long)p->total_k : (long long)p->batch * p->seqlen_k) == 0;
    if ((!no_q && (!h->q || !h->o || !h->dout || !h->lse || !h->dq)) || (!no_k && (!h->k || !h->v || !h->dk || !h->dv)))
      return ATTN_ERR_INVALID_ARG;
  }
  if (s == in || s == out || in == out) return ATTN_ERR_INVALID_ARG;
  // the staging buffers are contiguous (zero strides, or the contiguous ones spelt out)
  const bool group = p->cu_seqlens_q != nullptr;
  const TensorDesc t[8] = {{p->stride_q, p->seqlen_q, p->nhead_q, p->d_qk},   {p->stride_k, p->seqlen_k, p->nhead_kv, p->d_qk},
                           {p->stride_v, p->seqlen_k, p->nhead_kv, p->d_v},   {p->stride_o, p->seqlen_q, p->nhead_q, p->d_v},
                           {p->stride_dout, p->seqlen_q, p->nhead_q, p->d_v}, {p->stride_dq, p->seqlen_q, p->nhead_q, p->d_qk},
                           {p->stride_dk, p->seqlen_k, p->nhead_kv, p->d_qk}, {p->stride_dv, p->seqlen_k, p->nhead_kv, p->d_v}};
  for (const TensorDesc& x : t) {
    if (all_zero(x.in)) continue;
    const long long hs = x.dim, r = (long long)x.heads * x.dim, b = (long long)x.seqlen * r;
    if (x.in[1] != r || x.in[2] != hs || (!group && p->batch > 1 && x.in[0] != b)) return ATTN_ERR_INVALID_ARG;
  }
  attn_bwd_params e;
  Strides sx[8];
  if ((st = effective_bwd(*p, &e, sx)) != ATTN_OK) return st;
  if (!ws || ws_bytes < ws_layout(e).total) return ATTN_ERR_WORKSPACE_TOO_SMALL;
  // chunk grid: nbg runs of batch entries x nhg runs of kv heads
  const int nb = group ? 1 : p->batch, G = p->nhead_q / p->nhead_kv;
  if (chunks < 1) chunks = 1;
  if (chunks > 64) chunks = 64;
  int nbg = chunks < nb ? chunks : nb, nhg = 1;
  if (chunks > nb) {
    nhg = (chunks + nb - 1) / nb;
    if (nhg > p->nhead_kv) nhg = p->nhead_kv;
    if ((long long)nbg * nhg > 64) nhg = 64 / nbg > 0 ? 64 / nbg : 1;
  }
  const int nchunks = nbg * nhg;
  const size_t es = dtype_bytes(p->dtype);
  const long long rq = group ? p->total_q : p->seqlen_q, rk = group ? p->total_k : p->seqlen_k;
  // q, k, v, o, dout, dq, dk, dv; the kv-side tensors take kv-head ranges
  const HostTensor ht[8] = {{rq, p->nhead_q, p->d_qk, es},  {rk, p->nhead_kv, p->d_qk, es}, {rk, p->nhead_kv, p->d_v, es},
                            {rq, p->nhead_q, p->d_v, es},   {rq, p->nhead_q, p->d_v, es},   {rq, p->nhead_q, p->d_qk, es},
                            {rk, p->nhead_kv, p->d_qk, es}, {rk, p->nhead_kv, p->d_v, es}};
  const bool kv_side[8] = {false, true, true, false, false, false, true, true};
  const void* hsrc[5] = {h->q, h->k, h->v, h->o, h->dout};
  void* hdst[3] = {h->dq, h->dk, h->dv};
  const void* dptr[8] = {p->q, p->k, p->v, p->o, p->dout, p->dq, p->dk, p->dv};
  // per chunk: O, dO and LSE in (the preprocess reads only those), all inputs
  // in, main kernel done (dK, dV final), reduce/convert done (dQ final)
  enum { E_PRE, E_IN, E_MAIN, E_CONV, E_N };
  cudaEvent_t ev[64][E_N], ev_out;
  int made = 0;
  for (; made < nchunks; ++made) {
    int k = 0;
    while (k < E_N && cudaEventCreateWithFlags(&ev[made][k], cudaEventDisableTiming) == cudaSuccess) ++k;
    if (k < E_N) {
      while (k > 0) cudaEventDestroy(ev[made][--k]);
      break;
    }
  }
  const bool have_out = made == nchunks && cudaEventCreateWithFlags(&ev_out, cudaEventDisableTiming) == cudaSuccess;
  bool ok = have_out;
  // the caller's earlier work on `s` comes before the first copy
  if (ok) ok = cudaEventRecord(ev[0][E_CONV], s) == cudaSuccess && cudaStreamWaitEvent(in, ev[0][E_CONV], 0) == cudaSuccess &&
               cudaStreamWaitEvent(out, ev[0][E_CONV], 0) == cudaSuccess;
  for (int c = 0; ok && c < nchunks; ++c) {
    const int bg = c / nhg, hg = c % nhg;
    const int b0 = (int)((long long)nb * bg / nbg), b1 = (int)((long long)nb * (bg + 1) / nbg);
    const int k0 = (int)((long long)p->nhead_kv * hg / nhg), k1 = (int)((long long)p->nhead_kv * (hg + 1) / nhg);
    const int q0 = k0 * G, q1 = k1 * G;
    auto heads = [&](int i, int& x0, int& x1) { x0 = kv_side[i] ? k0 : q0; x1 = kv_side[i] ? k1 : q1; };
    auto copy_in = [&](int i) {
      int x0, x1;
      heads(i, x0, x1);
      return copy_part(ht[i], const_cast<void*>(dptr[i]), hsrc[i], b0, b1, x0, x1, cudaMemcpyHostToDevice, in);
    };
    // O, dO, then the LSE rows of the chunk: [b0, b1) x [q0, q1) x rows, one
    // block (either the heads are all of them or the chunk has one batch entry)
    ok = copy_in(3) && copy_in(4);
    const size_t lse_off = ((size_t)b0 * p->nhead_q + q0) * rq;
    const size_t lse_n = (size_t)(b1 - b0) * (q1 - q0) * rq;
    ok = ok && cudaMemcpyAsync(const_cast<float*>(p->lse) + lse_off, h->lse + lse_off, lse_n * sizeof(float),
                               cudaMemcpyHostToDevice, in) == cudaSuccess;
    ok = ok && cudaEventRecord(ev[c][E_PRE], in) == cudaSuccess;
    // then Q, K, V, which only the main kernel reads
    ok = ok && copy_in(0) && copy_in(1) && copy_in(2) && cudaEventRecord(ev[c][E_IN], in) == cudaSuccess;
    if (!ok) break;
    attn_bwd_params part = *p;
    if (!group) part.batch = b1 - b0;
    part.nhead_q = q1 - q0;
    part.nhead_kv = k1 - k0;
    void* views[8];
    for (int i = 0; i < 8; ++i) {
      int x0, x1;
      heads(i, x0, x1);
      const HostTensor& x = ht[i];
      views[i] = static_cast<char*>(const_cast<void*>(dptr[i])) +
                 ((size_t)b0 * x.rows * x.heads + x0) * x.dim * x.es;
      int64_t* sd[8] = {part.stride_q, part.stride_k, part.stride_v, part.stride_o,
                        part.stride_dout, part.stride_dq, part.stride_dk, part.stride_dv};
      sd[i][0] = (int64_t)x.rows * x.heads * x.dim;
      sd[i][1] = (int64_t)x.heads * x.dim;
      sd[i][2] = x.dim;
    }
    part.q = views[0]; part.k = views[1]; part.v = views[2]; part.o = views[3]; part.dout = views[4];
    part.dq = views[5]; part.dk = views[6]; part.dv = views[7];
    part.lse = p->lse + lse_off;
    Problem P;
    if ((st = prepare(&part, ws, ws_bytes, &P)) != ATTN_OK) break;
    if (empty_problem(P)) {
      if (!(ok = cudaStreamWaitEvent(s, ev[c][E_IN], 0) == cudaSuccess)) break;
      launch_empty(P, s, c > 0);
      if (!(ok = cudaEventRecord(ev[c][E_MAIN], s) == cudaSuccess)) break;
    } else {
      // the preprocess overlaps the copies of Q, K and V
      if (!(ok = cudaStreamWaitEvent(s, ev[c][E_PRE], 0) == cudaSuccess)) break;
      launch_schedule_preprocess(P, s, c > 0);
      if (!(ok = cudaStreamWaitEvent(s, ev[c][E_IN], 0) == cudaSuccess)) break;
      if ((st = launch_main(P, s)) != ATTN_OK) break;
      if (!(ok = cudaEventRecord(ev[c][E_MAIN], s) == cudaSuccess)) break;
      launch_reduce_convert(P, s);
    }
    if (!(ok = cudaEventRecord(ev[c][E_CONV], s) == cudaSuccess && cudaGetLastError() == cudaSuccess)) break;
    auto copy_out = [&](int i) {
      int x0, x1;
      heads(5 + i, x0, x1);
      return copy_part(ht[5 + i], hdst[i], dptr[5 + i], b0, b1, x0, x1, cudaMemcpyDeviceToHost, out);
    };
    // dK and dV come down while dQ is converted
    ok = cudaStreamWaitEvent(out, ev[c][E_MAIN], 0) == cudaSuccess && copy_out(1) && copy_out(2) &&
         cudaStreamWaitEvent(out, ev[c][E_CONV], 0) == cudaSuccess && copy_out(0);
  }
  // `s` completes only after the last gradients are back on the host
  if (ok && st == ATTN_OK)
    ok = cudaEventRecord(ev_out, out) == cudaSuccess && cudaStreamWaitEvent(s, ev_out, 0) == cudaSuccess;
  for (int i = 0; i < made; ++i)
    for (int k = 0; k < E_N; ++k) cudaEventDestroy(ev[i][k]);
  if (have_out) cudaEventDestroy(ev_out);
  if (st != ATTN_OK) return st;
  return ok ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace attn

using namespace attn;

extern "C" int attn_bwd_host(const attn_bwd_params* p, const attn_host_tensors* host, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream, cudaStream_t copy_in,
                             cudaStream_t copy_out, int chunks) {
  return run_host(p, host, workspace, workspace_bytes, stream, copy_in, copy_out, chunks);
}

extern "C" int attn_bwd_workspace_size(const attn_bwd_params* p, size_t* bytes) {
  if (!bytes) return ATTN_ERR_INVALID_ARG;
  *bytes = 0;
  const int st = validate_common(p);
  if (st != ATTN_OK) return st;
  if (p->deterministic < ATTN_DET_ATOMIC || p->deterministic > ATTN_DET_SPLIT) return ATTN_ERR_INVALID_ARG;
  attn_bwd_params e;
  Strides sx[8];
  const int s2 = effective_bwd(*p, &e, sx);
  if (s2 != ATTN_OK) return s2;
  *bytes = ws_layout(e).total;
  return ATTN_OK;
}

extern "C" int attn_bwd(const attn_bwd_params* p, void* workspace, size_t workspace_bytes,
                        cudaStream_t stream) {
  return run(p, workspace, workspace_bytes, stream, nullptr);
}

extern "C" int attn_bwd_timed(const attn_bwd_params* p, void* workspace, size_t workspace_bytes,
                              cudaStream_t stream, float stage_ms[4]) {
  if (!stage_ms) return ATTN_ERR_INVALID_ARG;
  int st = validate_bwd(p);
  if (st != ATTN_OK) return st;
  cudaEvent_t ev[4];
  for (int i = 0; i < 4; ++i)
    if (cudaEventCreate(&ev[i]) != cudaSuccess) return ATTN_ERR_CUDA;
  st = run(p, workspace, workspace_bytes, stream, ev);
  if (st == ATTN_OK) {
    if (cudaEventSynchronize(ev[3]) != cudaSuccess) st = ATTN_ERR_CUDA;
    cudaEventElapsedTime(&stage_ms[0], ev[0], ev[1]);
    cudaEventElapsedTime(&stage_ms[1], ev[1], ev[2]);
    cudaEventElapsedTime(&stage_ms[2], ev[2], ev[3]);
    cudaEventElapsedTime(&stage_ms[3], ev[0], ev[3]);
  }
  for (int i = 0; i < 4; ++i) cudaEventDestroy(ev[i]);
  return st;
}

extern "C" int attn_bwd_read_status(const void* workspace, cudaStream_t stream, int* status) {
  if (!workspace || !status) return ATTN_ERR_INVALID_ARG;
  int h[HDR_WORDS];
  if (cudaStreamSynchronize(stream) != cudaSuccess) return ATTN_ERR_CUDA;
  if (cudaMemcpy(h, workspace, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
  *status = h[HDR_STATUS];
  return ATTN_OK;
}

extern "C" int attn_fwd(const attn_fwd_params* p, cudaStream_t stream) {
  const int st = validate_fwd(p);
  if (st != ATTN_OK) return st;
  attn_fwd_params e;
  FwdLayout L;
  const int s2 = effective_fwd(*p, &e, &L);
  if (s2 != ATTN_OK) return s2;
  const bool gq = e.cu_seqlens_q != nullptr;
  if ((gq ? (long long)e.total_q : (long long)e.batch * e.seqlen_q) == 0) return ATTN_OK;   // no rows to write
  if ((gq ? (long long)e.total_k : (long long)e.batch * e.seqlen_k) == 0) {
    launch_fwd_no_keys(e, L, stream);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
  }
  // the tensor-core forward has no bias or dropout: the CUDA-core one takes those
  const bool extras = e.bias_type != ATTN_BIAS_NONE || e.dropout_p > 0.f;
  const int s3 = extras ? ATTN_ERR_UNSUPPORTED_HEADDIM : launch_fwd_tc(e, L, stream);
  if (s3 == ATTN_ERR_UNSUPPORTED_HEADDIM) launch_fwd(e, L, stream);   // fp32, other head dims, extras
  else if (s3 != ATTN_OK) return s3;
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

extern "C" const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED_HEADDIM: return "unsupported head dimension for this dtype";
    case ATTN_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case ATTN_ERR_CUDA: return "CUDA call failed";
    case ATTN_ERR_DEVICE_FLAG: return "device reported an error";
    case ATTN_ERR_TIMEOUT: return "bounded device wait expired";
    case ATTN_ERR_BAD_SEQLENS: return "cu_seqlens inconsistent with declared bounds";
    default: return "unknown status";
  }
}

extern "C" int attn_selftest_waits(void* scratch, size_t scratch_bytes, cudaStream_t stream, int status[3]) {
  if (!status) return ATTN_ERR_INVALID_ARG;
  return selftest_waits(scratch, scratch_bytes, stream, status);
}
