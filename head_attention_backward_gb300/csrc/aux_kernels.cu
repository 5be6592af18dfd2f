// Scheduler, preprocess and dQ reduce/convert kernels of the FMHA backward.
//
// * schedule: validates cu_seqlens on the device and writes the list of work
//   items (segment, kv head, KV tile) in KV-tile-major order, so the most
//   expensive causal tiles (lowest KV-tile index) are dealt first.  It replaces
//   the host-side seqstart copy CK's group-mode launcher needed (aiter PR
//   #2216 follow-up commit on the unified workspace: ".to(at::kCPU)").
// * preprocess: D = rowsum(dO * O) in fp32 and the negated log2-scaled LSE, plus the
//   zero-fill of the single atomic dq_acc slice (the "zero_init" the atomic
//   path requires, aiter PR #2216 follow-up: workspace_alloc(bytes, zero_init)).
// * reduce_convert: dQ = scale * sum over KV tiles of the dq_acc slices, in
//   ascending slice order, cast to the output dtype (the "dq_convert"
//   post-kernel of TransformerEngine PR #671, Summary, and the split
//   accumulation "converted back to final gradients" of aiter PR #2216).
#include "common.cuh"

namespace attn {

// ----------------------------------------------------------------- schedule

// Grouped work order (group mode only): used when the dq_acc slice exceeds
// SCHED_GROUP_ABOVE bytes, with groups of about SCHED_GROUP_BYTES of query
// tiles (L2 is 129 MB on GB300).  Measured on the packed THD workload (a
// 268 MB slice): main kernel 0.817 -> 0.668 ms in ordered mode; on batch
// workloads whose slice about fits L2, groups of one entry lengthened the
// fold's waits, so they keep the plain order.
constexpr long long SCHED_GROUP_ABOVE = 160LL << 20;
constexpr long long SCHED_GROUP_BYTES = 96LL << 20;
constexpr int SCHED_MAX_SEGS = 2048;   // segments cached in shared memory

// keep_status: a later part of one call split into parts (attn_bwd_host); the
// status of the earlier parts stays, and a part after a failed one does no work.
__global__ void __launch_bounds__(256) schedule_kernel(Problem P, int keep_status) {
  __shared__ int s_bad;
  __shared__ int s_lk[SCHED_MAX_SEGS], s_grp[SCHED_MAX_SEGS];
  __shared__ int s_cq[SCHED_MAX_SEGS + 1], s_ck[SCHED_MAX_SEGS + 1];
  const int tid = threadIdx.x;
  // the logical offsets are read many times below: one parallel pass copies
  // them into shared memory (up to SCHED_MAX_SEGS segments; beyond that they
  // are read from global memory)
  const bool cached = P.group && P.nseg <= SCHED_MAX_SEGS;
  if (cached) {
    for (int b = tid; b <= P.nseg; b += blockDim.x) {
      s_cq[b] = P.cu_q[b];
      s_ck[b] = P.cu_k[b];
    }
  }
  const int* cq = cached ? s_cq : P.cu_q;
  const int* ck = cached ? s_ck : P.cu_k;
  if (tid == 0) {
    s_bad = 0;
    if (keep_status && P.hdr[HDR_STATUS] != 0) {
      s_bad = 2;
    } else {
      P.hdr[HDR_STATUS] = 0;
      P.hdr[HDR_DIAG] = 0;
    }
    P.hdr[HDR_NEXT] = 0;
  }
  __syncthreads();
  if (s_bad == 0 && tid >= 16 && tid < HDR_WORDS) P.hdr[tid] = 0;   // optional per-site wait counters
  if (P.group && s_bad == 0) {
    // lengths from the logical offsets; each segment's physical rows
    // [start, start + length) lie before the next segment's start and inside
    // the tensor (without padding the starts are the offsets themselves and
    // the last one must equal the row total)
    for (int b = tid; b < P.nseg; b += blockDim.x) {
      const int lq = cq[b + 1] - cq[b], lk = ck[b + 1] - ck[b];
      bool bad = lq < 0 || lk < 0 || lq > P.sq || lk > P.sk;
      const long long sq0 = P.st_q[b], sq1 = P.st_q[b + 1];
      const long long sk0 = P.st_k[b], sk1 = P.st_k[b + 1];
      bad |= sq0 + lq > sq1 || sk0 + lk > sk1;
      if (b == 0) bad |= cq[0] != 0 || ck[0] != 0 || sq0 < 0 || sk0 < 0;
      if (b == P.nseg - 1) {
        bad |= sq1 > P.tq || sk1 > P.tk;
        if (P.st_q == P.cu_q) bad |= sq1 != P.tq;
        if (P.st_k == P.cu_k) bad |= sk1 != P.tk;
      }
      if (bad) s_bad = 1;
    }
  }
  __syncthreads();
  if (s_bad) {
    // no work items and no query tiles: nothing later in the call touches dQ
    // rows derived from the rejected cu_seqlens
    if (tid == 0) {
      if (s_bad == 1) P.hdr[HDR_STATUS] = ATTN_ERR_BAD_SEQLENS;
      P.hdr[HDR_NITEMS] = 0;
    }
    for (int b = tid; b <= P.nseg; b += blockDim.x) P.tile_off[b] = 0;
    return;
  }
  // Enumeration by warp 0, KV-tile-major: for kt, for segment, for kv head.
  // When the dq_acc slice is much larger than L2, consecutive segments are
  // first taken in groups of about SCHED_GROUP_BYTES of query tiles each (and
  // KV-tile-major inside a group), so that in ordered-fold mode the partial
  // sums a group adds into stay in L2 while its KV tiles pass over them.
  // Either way each segment's KV tiles stay in ascending order, which the
  // ordered fold's waits rely on.
  if (tid < 32) {
    const int lane = tid;
    const long long tile_bytes = (long long)P.hq * P.dqk * BM * 4;   // one query tile's partial sums, all heads
    const bool grouped = P.group && P.nseg <= SCHED_MAX_SEGS && (long long)P.ntiles * tile_bytes > SCHED_GROUP_ABOVE;
    int n = 0;
    auto emit = [&](int g0, int g1, int nkv, const int* lks) {
      for (int kt = 0; kt < nkv; ++kt) {
        for (int b0 = g0; b0 < g1; b0 += 32) {
          const int b = b0 + lane;
          bool has = false;
          if (b < g1) {
            const int lk = lks ? lks[b] : (P.group ? ck[b + 1] - ck[b] : P.sk);
            has = kt * BN < lk;
          }
          const unsigned m = __ballot_sync(0xffffffffu, has);
          const int before = __popc(m & ((1u << lane) - 1u));
          if (has) {
            const int base = n + before * P.hkv;
            for (int h = 0; h < P.hkv; ++h)
              if (base + h < P.max_items) P.items[base + h] = make_int4(b, h, kt, 0);
          }
          n += __popc(m) * P.hkv;
        }
      }
    };
    if (!grouped) {
      emit(0, P.nseg, cdiv(P.sk > 0 ? P.sk : 1, BN), nullptr);
    } else {
      // segment lengths and group ids (query-tile bytes before the segment /
      // SCHED_GROUP_BYTES) into shared memory, 32 segments at a time
      long long carry = 0;
      for (int b0 = 0; b0 < P.nseg; b0 += 32) {
        const int b = b0 + lane;
        int lq = 0, lk = 0;
        if (b < P.nseg) {
          lq = cq[b + 1] - cq[b];
          lk = ck[b + 1] - ck[b];
        }
        const long long bytes = (long long)cdiv(max(lq, 0), BM) * tile_bytes;
        long long incl = bytes;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const long long y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        if (b < P.nseg) {
          s_lk[b] = max(lk, 0);
          s_grp[b] = (int)((carry + incl - bytes) / SCHED_GROUP_BYTES);
        }
        carry += __shfl_sync(0xffffffffu, incl, 31);
      }
      __syncwarp();
      for (int g0 = 0; g0 < P.nseg;) {
        int g1 = g0 + 1, nkv = cdiv(s_lk[g0], BN);
        while (g1 < P.nseg && s_grp[g1] == s_grp[g0]) nkv = max(nkv, cdiv(s_lk[g1++], BN));
        emit(g0, g1, nkv, s_lk);
        g0 = g1;
      }
    }
    if (lane == 0) {
      if (n > P.max_items) {
        P.hdr[HDR_STATUS] = ATTN_ERR_BAD_SEQLENS;
        n = 0;
      }
      P.hdr[HDR_NITEMS] = n;
    }
  } else if (tid < 64 && P.group) {
    // warp 1: first dq_acc query-tile index of every segment (exclusive scan
    // of ceil(Lq_b / BM)); dq_acc holds P.ntiles tiles per (slice, head)
    const int lane = tid - 32;
    int base = 0;
    for (int b0 = 0; b0 <= P.nseg; b0 += 32) {
      const int b = b0 + lane;
      int v = 0;
      if (b < P.nseg) v = cdiv(cq[b + 1] - cq[b], BM);
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (b <= P.nseg) P.tile_off[b] = base + incl - v;
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0 && base > P.ntiles) P.hdr[HDR_STATUS] = ATTN_ERR_BAD_SEQLENS;
  }
}


// --------------------------------------------------------------- preprocess
// D and -LSE*log2(e) of every (packed token, query head) row.  16-bit
// inputs: half a warp per group of four rows, 16-byte loads of O and dO, one
// resident wave of blocks.  fp32 inputs: one warp per row.  In atomic and
// ordered-fold modes the single dq_acc slice is zeroed as well.

// Index in the LSE layout of row r = token * Hq + head of O / dO.
__device__ __forceinline__ long long lse_index(const Problem& P, long long r) {
  const long long tok = r / P.hq;
  const int h = (int)(r - tok * P.hq);
  if (P.group) return (long long)h * P.tq + tok;
  const long long b = tok / P.sq, q = tok - b * P.sq;
  return (b * P.hq + h) * P.sq + q;
}

__device__ __forceinline__ void store_row_stats(const Problem& P, long long li, float l, float acc) {
  const float LOG2E = 1.4426950408889634f;
  P.dvec[li] = acc;
  P.nlse2[li] = (l == -INFINITY) ? -INFINITY : -l * LOG2E;
}

__device__ __forceinline__ void write_row_stats(const Problem& P, long long r, float acc) {
  const long long li = lse_index(P, r);
  if (!ATTN_INDEX_OK(P, li >= 0 && li < P.n_lse, 8)) return;
  store_row_stats(P, li, P.lse[li], acc);
}

__device__ __forceinline__ float dot8(uint4 a, uint4 b, __nv_bfloat16*) {
  const __nv_bfloat162* x = reinterpret_cast<const __nv_bfloat162*>(&a);
  const __nv_bfloat162* y = reinterpret_cast<const __nv_bfloat162*>(&b);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 u = __bfloat1622float2(x[i]), v = __bfloat1622float2(y[i]);
    s = fmaf(u.x, v.x, s);
    s = fmaf(u.y, v.y, s);
  }
  return s;
}

__device__ __forceinline__ float dot8(uint4 a, uint4 b, __half*) {
  const __half2* x = reinterpret_cast<const __half2*>(&a);
  const __half2* y = reinterpret_cast<const __half2*>(&b);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 u = __half22float2(x[i]), v = __half22float2(y[i]);
    s = fmaf(u.x, v.x, s);
    s = fmaf(u.y, v.y, s);
  }
  return s;
}

// Padded group layout: gradient rows that belong to no segment are zero.
// Gap g in [0, nseg] holds the rows from the end of segment g-1 (row 0 for
// g = 0) up to the start of segment g (the row total for g = nseg); the
// schedule kernel has checked that the gaps are well formed.  A (row, head)
// vector of `dim` elements is a whole number of 4-byte words at a word
// boundary for every supported dtype, head dim and stride.
__device__ void zero_padding_rows(const int* st, const int* cu, int nseg, int total, int heads, int dim,
                                  const Strides& x, int esize, void* out) {
  const int wpv = dim * esize / 4;   // words per (row, head)
  uint32_t* o = static_cast<uint32_t*>(out);
  for (int g = blockIdx.x; g <= nseg; g += gridDim.x) {
    const long long a = g == 0 ? 0 : (long long)st[g - 1] + (cu[g] - cu[g - 1]);
    const long long e = g == nseg ? total : st[g];
    const long long n = (e - a) * heads * wpv;
    for (long long i = threadIdx.x; i < n; i += blockDim.x) {
      const long long rr = i / ((long long)heads * wpv);
      const int rem = (int)(i - rr * heads * wpv), hh = rem / wpv, wd = rem - hh * wpv;
      o[elem_off(x, a + rr, hh) * esize / 4 + wd] = 0u;
    }
  }
}

// Rows [0, rows) x heads of a strided gradient tensor set to zero (each
// (row, head) vector a whole number of 4-byte words at a word boundary).
__device__ void zero_all_rows(long long rows, int heads, int dim, const Strides& x, int esize, void* out) {
  const int wpv = dim * esize / 4;
  uint32_t* o = static_cast<uint32_t*>(out);
  const long long n = rows * heads * wpv;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const long long rr = i / ((long long)heads * wpv);
    const int rem = (int)(i - rr * heads * wpv), hh = rem / wpv, wd = rem - hh * wpv;
    o[elem_off(x, rr, hh) * esize / 4 + wd] = 0u;
  }
}

// No keys at all: every query row sees nothing, dQ = 0.  No queries at all:
// no key is seen, dK = dV = 0.
__global__ void __launch_bounds__(256) empty_problem_kernel(Problem P, int keep_status) {
  if (blockIdx.x == 0 && !keep_status)
    for (int i = threadIdx.x; i < HDR_WORDS; i += blockDim.x) P.hdr[i] = 0;
  const int w = P.dtype == ATTN_FP32 ? 4 : 2;
  if (rows_k(P) == 0) zero_all_rows(rows_q(P), P.hq, P.dqk, P.sdq_, w, P.dq);
  if (rows_q(P) == 0) {
    zero_all_rows(rows_k(P), P.hkv, P.dqk, P.sdk_, w, P.dk);
    zero_all_rows(rows_k(P), P.hkv, P.dv, P.sdv_, w, P.dv_out);
  }
}

void launch_empty(const Problem& P, cudaStream_t st, bool keep_status) {
  empty_problem_kernel<<<256, 256, 0, st>>>(P, keep_status ? 1 : 0);
}

constexpr int PRE_BLOCKS_PER_SM = 3;

// Batch mode needs no cu_seqlens validation, so the preprocess kernel also
// does the scheduler's part (sched != 0): block 0 resets the workspace header
// (keeping an earlier part's failure when sched == 2, as schedule_kernel
// does) and the grid writes the work list in the same KV-tile-major order,
// item (kt, b, h) at index (kt * B + b) * Hkv + h.  This saves the one-block
// scheduler launch.  The main kernel starts after this kernel has finished,
// so it sees the header and the list complete.
__device__ __forceinline__ void batch_schedule(const Problem& P, int sched, long long tid, long long nthreads) {
  if (blockIdx.x == 0) {
    __shared__ int s_skip;
    if (threadIdx.x == 0) {
      s_skip = sched == 2 && P.hdr[HDR_STATUS] != 0;
      if (!s_skip) {
        P.hdr[HDR_STATUS] = 0;
        P.hdr[HDR_DIAG] = 0;
      }
      P.hdr[HDR_NEXT] = 0;
      P.hdr[HDR_NITEMS] = s_skip ? 0 : P.max_items;
    }
    __syncthreads();
    if (!s_skip && threadIdx.x >= 16 && threadIdx.x < HDR_WORDS) P.hdr[threadIdx.x] = 0;
  }
  const int per_kt = P.nseg * P.hkv;
  for (long long i = tid; i < P.max_items; i += nthreads) {
    const int kt = (int)(i / per_kt), r = (int)(i - (long long)kt * per_kt);
    const int b = r / P.hkv;
    P.items[i] = make_int4(b, r - b * P.hkv, kt, 0);
  }
}

// VW: 16-byte vectors per lane and row (1 for d_v <= 128, 2 for d_v = 256).
template <typename T, int VW>
__global__ void __launch_bounds__(256, PRE_BLOCKS_PER_SM) preprocess_kernel(Problem P, long long ntok, int sched) {
  const int lane = threadIdx.x & 31;
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long nthreads = (long long)gridDim.x * blockDim.x;
  if (sched) batch_schedule(P, sched, tid, nthreads);
  const long long nrows = ntok * P.hq;
  if constexpr (sizeof(T) == 2) {
    // A half warp takes RPH consecutive rows at a time (16-byte loads; d_v and
    // every stride are multiples of 8; d_v is at most 128, one load per lane
    // and row, or 256, two).  All loads of a group, LSE included, are issued
    // before the first reduction so that each half warp keeps RPH rows in flight.
    constexpr int RPH = 4 / VW;
    const int sub = lane & 15;
    const long long hw = tid >> 4, nhw = nthreads >> 4;
    const uint4* O = static_cast<const uint4*>(P.o);
    const uint4* dO = static_cast<const uint4*>(P.dout);
    const int nv = P.dv / 8;
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    // the trip count is warp-uniform (the shuffles below take the full mask)
    for (long long w0 = (hw >> 1) * 2 * RPH; w0 < nrows; w0 += nhw * RPH) {
      const long long r0 = w0 + (hw & 1) * RPH;
      uint4 a[RPH], b[RPH], a2[VW == 2 ? RPH : 1], b2[VW == 2 ? RPH : 1];
      long long li[RPH];
      float l[RPH];
      // (token, head) and, in batch mode, (batch, query) of the first row by
      // division, of the next rows by stepping
      long long tok = r0 / P.hq;
      int h = (int)(r0 - tok * P.hq);
      long long bq = P.group ? 0 : tok / P.sq;
      long long q = tok - bq * P.sq;
      // element offsets of the row in O and dO (multiples of 8, non-negative)
      long long oo = elem_off(P.so_, tok, h), od = elem_off(P.sdo_, tok, h);
#pragma unroll
      for (int i = 0; i < RPH; ++i) {
        const long long r = r0 + i;
        const bool ok = r < nrows && sub < nv;
        a[i] = ok ? __ldcs(O + (oo >> 3) + sub) : z;
        b[i] = ok ? __ldcs(dO + (od >> 3) + sub) : z;
        if constexpr (VW == 2) {   // d_v = 256: the second half of the row
          const bool ok2 = r < nrows && sub + 16 < nv;
          a2[i] = ok2 ? __ldcs(O + (oo >> 3) + sub + 16) : z;
          b2[i] = ok2 ? __ldcs(dO + (od >> 3) + sub + 16) : z;
        }
        li[i] = P.group ? (long long)h * P.tq + tok : (bq * P.hq + h) * P.sq + q;
        l[i] = (sub == 0 && r < nrows && ATTN_INDEX_OK(P, li[i] >= 0 && li[i] < P.n_lse, 8)) ? P.lse[li[i]] : 0.f;
        if (++h == P.hq) {
          h = 0;
          ++tok;
          if (++q == P.sq) { q = 0; ++bq; }
          oo = elem_off(P.so_, tok, 0);
          od = elem_off(P.sdo_, tok, 0);
        } else {
          oo += P.so_.h;
          od += P.sdo_.h;
        }
      }
#pragma unroll
      for (int i = 0; i < RPH; ++i) {
        float acc = dot8(a[i], b[i], (T*)nullptr);
        if constexpr (VW == 2) acc += dot8(a2[i], b2[i], (T*)nullptr);
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (sub == 0 && r0 + i < nrows && li[i] >= 0 && li[i] < P.n_lse) store_row_stats(P, li[i], l[i], acc);
      }
    }
  } else {
    const long long warp = tid >> 5, nwarps = nthreads >> 5;
    const T* O = static_cast<const T*>(P.o);
    const T* dO = static_cast<const T*>(P.dout);
    for (long long r = warp; r < nrows; r += nwarps) {
      const long long tok = r / P.hq;
      const int h = (int)(r - tok * P.hq);
      const T* o = O + elem_off(P.so_, tok, h);
      const T* d = dO + elem_off(P.sdo_, tok, h);
      float acc = 0.f;
      for (int c = lane; c < P.dv; c += 32) acc += TypeOps<T>::to_f(o[c]) * TypeOps<T>::to_f(d[c]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) write_row_stats(P, r, acc);
    }
  }
  if (P.padded && *(volatile const int*)(P.hdr + HDR_STATUS) == 0) {
    const int w = (int)sizeof(T);
    zero_padding_rows(P.st_q, P.cu_q, P.nseg, P.tq, P.hq, P.dqk, P.sdq_, w, P.dq);
    zero_padding_rows(P.st_k, P.cu_k, P.nseg, P.tk, P.hkv, P.dqk, P.sdk_, w, P.dk);
    zero_padding_rows(P.st_k, P.cu_k, P.nseg, P.tk, P.hkv, P.dv, P.sdv_, w, P.dv_out);
  }
  if (!P.det || P.fold) {   // the single slice that partials are added into starts at zero
    float4* acc4 = reinterpret_cast<float4*>(P.dq_acc);
    const long long n4 = (long long)P.hq * P.ntiles * P.dqk * BM / 4;
    for (long long i = tid; i < n4; i += nthreads) acc4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (P.fold) {
    // ordered fold: no partial folded yet, and the first KV tile reaching
    // each query tile (a partial's rank is its KV tile minus that one)
    const long long n = (long long)tc_passes(P.dqk) * P.hq * P.ntiles;
    for (long long i = tid; i < n; i += nthreads) P.turn[i] = 0u;
    for (long long t = tid; t < P.ntiles; t += nthreads) {
      int b, qt, k = -1;
      if (tile_coords(P, (int)t, b, qt)) {
        const Seg sg = segment(P, b);
        k = first_kv_tile(mask_args(P.mask, P.left, P.right, sg.lq, sg.lk), sg.lq, sg.lk, qt);
      }
      P.klo[t] = k;
    }
  }
}

static int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

// dbias [B, Hq, Sq, Sk] (batch mode, attention bias with its gradient): the
// main kernel writes the rows of every (query tile, KV tile) pair it visits,
// masked entries as zeros; this kernel zeroes the pairs that no KV tile's
// query range reaches, one tile row (up to BN elements) per thread.
template <typename T>
__global__ void __launch_bounds__(256) dbias_fill_kernel(Problem P) {
  const MaskArgs m = mask_args(P.mask, P.left, P.right, P.sq, P.sk);
  const int ntq = cdiv(P.sq, BM), nkv = cdiv(P.sk, BN);
  const long long rows = (long long)P.nseg * P.hq * ntq * nkv * BM;
  T* db = static_cast<T*>(P.dbias);
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < rows; i += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(i % BM);
    long long t = i / BM;
    const int kt = (int)(t % nkv);
    t /= nkv;
    const int qt = (int)(t % ntq);
    const long long bh = t / ntq;
    const int q = qt * BM + r;
    if (q >= P.sq) continue;
    int lo, hi;
    qtile_range(m, P.sq, P.sk, kt, lo, hi);
    if (qt >= lo && qt < hi) continue;   // visited: the main kernel writes it
    T* row = db + (bh * P.sq + q) * P.sk + (long long)kt * BN;
    const int n = min(BN, P.sk - kt * BN);
    for (int c = 0; c < n; ++c) row[c] = TypeOps<T>::from_f(0.f);
  }
}

// sched: 0 = the scheduler kernel ran before; 1 / 2 = batch mode, this
// kernel schedules (2: keep an earlier part's status).
static void launch_preprocess_sched(const Problem& P, cudaStream_t st, int sched) {
  const long long ntok = P.group ? (long long)P.tq : (long long)P.nseg * P.sq;
  const int grid = num_sms() * PRE_BLOCKS_PER_SM;   // one resident wave
  const bool wide = P.dv > 128;
  switch (P.dtype) {
    case ATTN_BF16:
      if (wide) preprocess_kernel<__nv_bfloat16, 2><<<grid, 256, 0, st>>>(P, ntok, sched);
      else preprocess_kernel<__nv_bfloat16, 1><<<grid, 256, 0, st>>>(P, ntok, sched);
      break;
    case ATTN_FP16:
      if (wide) preprocess_kernel<__half, 2><<<grid, 256, 0, st>>>(P, ntok, sched);
      else preprocess_kernel<__half, 1><<<grid, 256, 0, st>>>(P, ntok, sched);
      break;
    default: preprocess_kernel<float, 1><<<grid, 256, 0, st>>>(P, ntok, sched); break;
  }
}

void launch_preprocess(const Problem& P, cudaStream_t st) { launch_preprocess_sched(P, st, 0); }

// Schedule + preprocess of one call (or one part of a call split into parts,
// keep_status: the earlier parts' status stays).  Group mode validates
// cu_seqlens in the scheduler kernel first; batch mode folds the schedule into
// the preprocess kernel (debug builds keep the separate scheduler, whose
// header reset then precedes every index check of the preprocess).
void launch_schedule_preprocess(const Problem& P, cudaStream_t st, bool keep_status) {
  if (P.dbias != nullptr) {
    const int grid = num_sms() * 4;
    if (P.dtype == ATTN_FP16) dbias_fill_kernel<__half><<<grid, 256, 0, st>>>(P);
    else dbias_fill_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(P);
  }
#ifndef ATTN_DEBUG
  if (!P.group) {
    launch_preprocess_sched(P, st, keep_status ? 2 : 1);
    return;
  }
#endif
  schedule_kernel<<<1, 256, 0, st>>>(P, keep_status ? 1 : 0);
  launch_preprocess_sched(P, st, 0);
}

// ----------------------------------------------------------- reduce/convert
// One block per (query head, query tile) at a time; one resident wave of
// blocks loops over the pairs.  Split mode: the query-major dQ
// tiles of the slices whose KV tile reaches this query tile (the others were
// never written) are summed in ascending slice order; atomic and ordered-fold
// modes read the single slice.  Each thread owns four consecutive d of one
// query row, so the scaled sum goes straight to dQ without a transpose.

constexpr int RC_THREADS = 256;

// NACC = float4 accumulators per thread = ceil(d_qk * BM / 4 / RC_THREADS).
// One (head, query tile) of the dQ output: w = head * ntiles + tile.
template <typename T, int NACC, bool SPLIT>
__device__ __forceinline__ void reduce_convert_tile(const Problem& P, long long w) {
  const int dqk = P.dqk;
  const int nv4 = dqk * BM / 4;      // float4 per dQ tile
  T* dQ = static_cast<T*>(P.dq);
  const int h = (int)(w / P.ntiles);
  const int t = (int)(w % P.ntiles);
  int b, qt;
  if (!tile_coords(P, t, b, qt)) return;   // beyond the last segment's tiles
  const Seg s = segment(P, b);
  const int nvalid = min(BM, s.lq - qt * BM);
  if (nvalid <= 0) return;
  float4 acc[NACC];
#pragma unroll
  for (int i = 0; i < NACC; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  // acc += tile a, then acc += tile b (b may be null); both tiles' loads are
  // issued before the first add, the order of the additions stays a then b
  auto add_tiles = [&](const float* a, const float* bt) {
    float4 xa[NACC], xb[NACC];
#pragma unroll
    for (int i = 0; i < NACC; ++i) {
      const int v = threadIdx.x + i * RC_THREADS;
      xa[i] = v < nv4 ? __ldcs(reinterpret_cast<const float4*>(a) + v) : make_float4(0.f, 0.f, 0.f, 0.f);
      xb[i] = (bt && v < nv4) ? __ldcs(reinterpret_cast<const float4*>(bt) + v) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < NACC; ++i) {
      acc[i].x += xa[i].x; acc[i].y += xa[i].y; acc[i].z += xa[i].z; acc[i].w += xa[i].w;
    }
    if (bt) {
#pragma unroll
      for (int i = 0; i < NACC; ++i) {
        acc[i].x += xb[i].x; acc[i].y += xb[i].y; acc[i].z += xb[i].z; acc[i].w += xb[i].w;
      }
    }
  };
  if constexpr (SPLIT) {
    const MaskArgs m = mask_args(P.mask, P.left, P.right, s.lq, s.lk);
    int nkv = cdiv(s.lk, BN);
    if (nkv > P.nsplits) nkv = P.nsplits;   // guards cu_seqlens that broke their bound
    // the slices whose KV tile reaches query tile qt, two at a time, ascending
    auto next = [&](int kt) {
      for (; kt < nkv; ++kt) {
        int lo, hi;
        qtile_range(m, s.lq, s.lk, kt, lo, hi);
        if (qt >= lo && qt < hi) break;
      }
      return kt;
    };
    for (int k0 = next(0); k0 < nkv;) {
      if constexpr (NACC > 8) {
        // d_qk = 256: one slice in flight at a time (register budget)
        if (ATTN_INDEX_OK(P, k0 < P.nsplits && t < P.ntiles, 10)) add_tiles(dq_tile(P, k0, h, t), nullptr);
        k0 = next(k0 + 1);
      } else {
        const int k1 = next(k0 + 1);
        if (ATTN_INDEX_OK(P, k0 < P.nsplits && t < P.ntiles, 10))
          add_tiles(dq_tile(P, k0, h, t), k1 < nkv ? dq_tile(P, k1, h, t) : nullptr);
        k0 = k1 < nkv ? next(k1 + 1) : nkv;
      }
    }
  } else if (s.lk > 0) {   // atomic and ordered fold: the single, pre-zeroed slice
#pragma unroll
    for (int i = 0; i < NACC; ++i) {
      const int v = threadIdx.x + i * RC_THREADS;
      if (v < nv4) acc[i] = __ldcs(reinterpret_cast<const float4*>(dq_tile(P, 0, h, t)) + v);
    }
  }
  T* dQt = dQ + elem_off(P.sdq_, s.q0 + qt * BM, h);   // row 0 of the tile
#pragma unroll
  for (int i = 0; i < NACC; ++i) {
    const int v = threadIdx.x + i * RC_THREADS;
    const int c = (4 * v) / dqk, e = (4 * v) - c * dqk;   // query row, first d
    if (v < nv4 && c < nvalid &&
        ATTN_INDEX_OK(P, s.q0 + qt * BM + c >= 0 && s.q0 + qt * BM + c < rows_q(P) && h < P.hq, 9)) {
      T* row = dQt + c * P.sdq_.r + e;
      T o4[4] = {TypeOps<T>::from_f(acc[i].x * P.scale), TypeOps<T>::from_f(acc[i].y * P.scale),
                 TypeOps<T>::from_f(acc[i].z * P.scale), TypeOps<T>::from_f(acc[i].w * P.scale)};
      if (sizeof(T) == 2) {
        *reinterpret_cast<uint2*>(row) = *reinterpret_cast<uint2*>(o4);
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) row[k] = o4[k];
      }
    }
  }
}

// SPLIT: sum the split slices (deterministic split mode); otherwise convert
// the single slice (atomic, ordered fold), an instantiation of its own so that
// its lower register count allows a full SM of blocks.
template <typename T, int NACC, bool SPLIT>
__global__ void __launch_bounds__(RC_THREADS) reduce_convert_kernel(Problem P) {
  // a rejected problem (bad cu_seqlens, expired wait) leaves dQ untouched
  if (*(volatile const int*)(P.hdr + HDR_STATUS) != 0) return;
  const long long work = (long long)P.hq * P.ntiles;
  // one resident wave of blocks walks the (head, tile) pairs head-major
  for (long long w = blockIdx.x; w < work; w += gridDim.x) reduce_convert_tile<T, NACC, SPLIT>(P, w);
}

// Single slice: one resident wave of blocks (as many as the occupancy of the
// instantiation allows on every SM), or fewer when there are fewer (head,
// tile) pairs.  Split slices: one block per pair (a block sums a variable
// number of slices, so many independent blocks overlap better than a loop).
template <typename K>
static void launch_rc_kernel(K kern, const Problem& P, long long work, bool wave_grid, cudaStream_t st) {
  long long grid = work;
  if (wave_grid) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, RC_THREADS, 0) != cudaSuccess || per_sm < 1)
      per_sm = 1;
    const long long wave = (long long)num_sms() * per_sm;
    if (wave < grid) grid = wave;
  }
  kern<<<(unsigned)grid, RC_THREADS, 0, st>>>(P);
}

template <typename T, bool SPLIT>
static void launch_rc(const Problem& P, long long work, cudaStream_t st) {
  const int nacc = cdiv(P.dqk * BM / 4, RC_THREADS);
  if (nacc <= 4) launch_rc_kernel(reduce_convert_kernel<T, 4, SPLIT>, P, work, !SPLIT, st);
  else if (nacc <= 8) launch_rc_kernel(reduce_convert_kernel<T, 8, SPLIT>, P, work, !SPLIT, st);
  else if (nacc <= 12) launch_rc_kernel(reduce_convert_kernel<T, 12, SPLIT>, P, work, !SPLIT, st);
  else launch_rc_kernel(reduce_convert_kernel<T, 16, SPLIT>, P, work, !SPLIT, st);
}

template <typename T>
static void launch_rc(const Problem& P, long long work, cudaStream_t st) {
  if (P.det && !P.fold) launch_rc<T, true>(P, work, st);
  else launch_rc<T, false>(P, work, st);
}

void launch_reduce_convert(const Problem& P, cudaStream_t st) {
  const long long work = (long long)P.hq * P.ntiles;   // (head, query tile) pairs
  if (work <= 0) return;
  switch (P.dtype) {
    case ATTN_BF16: launch_rc<__nv_bfloat16>(P, work, st); break;
    case ATTN_FP16: launch_rc<__half>(P, work, st); break;
    default: launch_rc<float>(P, work, st); break;
  }
}

}  // namespace attn
