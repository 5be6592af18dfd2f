// SIMT (CUDA-core, fp32 arithmetic) kernels:
//
// * fwd_kernel: the forward helper that produces O and the natural-log LSE
//   for benchmark and test inputs (the forward implied by ck_attn_fwd in
//   TransformerEngine PR #446).  Online softmax over 64-key tiles.
// * bwd_simt_kernel: the backward pass for fp32 inputs.  It runs the same
//   KV-tile-major decomposition, work list, dq_acc layout and dQ reduction as
//   the tensor-core kernel, with one thread per key row.
#include "common.cuh"

namespace attn {

// ------------------------------------------------------------------ forward

constexpr int FWD_BQ = 64;   // query rows per block
constexpr int FWD_BK = 64;   // keys per tile
constexpr int FWD_THREADS = 256;

// NC: output columns per thread (d_v <= 4 NC).
template <typename T, int NC>
__global__ void __launch_bounds__(FWD_THREADS) fwd_kernel(attn_fwd_params p, FwdLayout L, int group) {
  extern __shared__ float smem[];
  const int dqk = p.d_qk, dv = p.d_v;
  const int sq_stride = dqk + 1, sk_stride = dqk + 1, sv_stride = dv;
  float* sQ = smem;                          // [FWD_BQ][dqk+1]
  float* sK = sQ + FWD_BQ * sq_stride;       // [FWD_BK][dqk+1]
  float* sV = sK + FWD_BK * sk_stride;       // [FWD_BK][dv]
  float* sP = sV + FWD_BK * sv_stride;       // [FWD_BQ][FWD_BK+1]

  const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int g = p.nhead_q / p.nhead_kv, hk = h / g;
  int q0, lq, k0, lk;
  if (group) {
    lq = p.cu_seqlens_q[b + 1] - p.cu_seqlens_q[b];
    lk = p.cu_seqlens_k[b + 1] - p.cu_seqlens_k[b];
    q0 = p.cu_seqlens_q_padded ? p.cu_seqlens_q_padded[b] : p.cu_seqlens_q[b];
    k0 = p.cu_seqlens_k_padded ? p.cu_seqlens_k_padded[b] : p.cu_seqlens_k[b];
  } else {
    q0 = b * p.seqlen_q; lq = p.seqlen_q; k0 = b * p.seqlen_k; lk = p.seqlen_k;
  }
  const int qs = qt * FWD_BQ;
  if (qs >= lq) return;
  const T* Q = static_cast<const T*>(p.q);
  const T* K = static_cast<const T*>(p.k);
  const T* V = static_cast<const T*>(p.v);
  T* O = static_cast<T*>(p.o);
  const int tid = threadIdx.x;
  for (int i = tid; i < FWD_BQ * dqk; i += FWD_THREADS) {
    const int r = i / dqk, c = i % dqk;
    float x = 0.f;
    if (qs + r < lq) x = TypeOps<T>::to_f(Q[elem_off(L.q, q0 + qs + r, h) + c]);
    sQ[r * sq_stride + c] = x;
  }
  const MaskArgs m = mask_args(p.mask, p.window_left, p.window_right, lq, lk);
  // attention bias (batch mode) and dropout: bh = b * Hq + h indexes the
  // dropout counter, the caller's (batch entry, head) the bias
  const T* bias = static_cast<const T*>(p.bias);
  const long long bias_off = bias ? (long long)(b + h / L.hq0) * L.bias_sb + (long long)(h % L.hq0) * L.bias_sh : 0;
  const uint32_t bh = (uint32_t)(b * p.nhead_q + h);
  const bool drop = p.dropout_p > 0.f;
  unsigned long long seed = 0, offset = 0;
  uint32_t thr = 0;
  float dscale = 1.f;
  if (drop) {
    seed = *p.philox_seed;
    offset = *p.philox_offset;
    const double t = floor((double)p.dropout_p * 4294967296.0);
    thr = t >= 4294967295.0 ? 4294967295u : (uint32_t)t;
    dscale = 1.f / (1.f - p.dropout_p);
  }
  // keys any row of this tile can see
  const int qe = min(qs + FWD_BQ, lq) - 1;
  long long klo = 0, khi = (long long)lk - 1;
  if (m.left >= 0) klo = max(klo, (long long)qs + m.off - m.left);
  if (m.right >= 0) khi = min(khi, (long long)qe + m.off + m.right);

  const int row = tid >> 2, sub = tid & 3;
  const int ncol = (dv + 3) / 4;   // output columns of this thread: sub, sub+4, ...
  float acc[NC];
#pragma unroll
  for (int i = 0; i < NC; ++i) acc[i] = 0.f;
  float mrow = -INFINITY, lrow = 0.f;
  const float sl2 = p.softmax_scale * 1.4426950408889634f;

  for (long long kb = (klo / FWD_BK) * FWD_BK; kb <= khi; kb += FWD_BK) {
    __syncthreads();
    for (int i = tid; i < FWD_BK * dqk; i += FWD_THREADS) {
      const int r = i / dqk, c = i % dqk;
      const long long kk = kb + r;
      sK[r * sk_stride + c] = kk < lk ? TypeOps<T>::to_f(K[elem_off(L.k, k0 + kk, hk) + c]) : 0.f;
    }
    for (int i = tid; i < FWD_BK * dv; i += FWD_THREADS) {
      const int r = i / dv, c = i % dv;
      const long long kk = kb + r;
      sV[r * sv_stride + c] = kk < lk ? TypeOps<T>::to_f(V[elem_off(L.v, k0 + kk, hk) + c]) : 0.f;
    }
    __syncthreads();
    float s[FWD_BK / 4];
    float tmax = -INFINITY;
    const int qi = qs + row;
#pragma unroll
    for (int t = 0; t < FWD_BK / 4; ++t) {
      const int j = sub + 4 * t;
      const long long kk = kb + j;
      float x = 0.f;
      for (int c = 0; c < dqk; ++c) x += sQ[row * sq_stride + c] * sK[j * sk_stride + c];
      const bool ok = qi < lq && kk < lk && visible(m, qi, (int)kk);
      if (ok && bias) x = fmaf(TypeOps<T>::to_f(bias[bias_off + (long long)qi * p.seqlen_k + kk]), 1.f / p.softmax_scale, x);
      s[t] = ok ? x * sl2 : -INFINITY;
      tmax = fmaxf(tmax, s[t]);
    }
    tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
    tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
    const float mnew = fmaxf(mrow, tmax);
    float psum = 0.f;
    if (mnew == -INFINITY) {
#pragma unroll
      for (int t = 0; t < FWD_BK / 4; ++t) sP[row * (FWD_BK + 1) + sub + 4 * t] = 0.f;
    } else {
      const float corr = fast_exp2(mrow - mnew);
      lrow *= corr;
      for (int i = 0; i < ncol; ++i) acc[i] *= corr;
#pragma unroll
      for (int t = 0; t < FWD_BK / 4; ++t) {
        const float e = fast_exp2(s[t] - mnew);
        psum += e;
        float ev = e;
        if (drop) {   // the row sum keeps every weight, the product with V only the kept ones
          const long long kk = kb + sub + 4 * t;
          const uint32_t bits = dropout_keep4(seed, offset, (uint32_t)(qi >> 2), (uint32_t)kk, bh, thr);
          ev = ((bits >> (qi & 3)) & 1u) ? e * dscale : 0.f;
        }
        sP[row * (FWD_BK + 1) + sub + 4 * t] = ev;
      }
      mrow = mnew;
    }
    lrow += psum;
    __syncwarp();
    for (int i = 0; i < ncol; ++i) {
      const int c = sub + 4 * i;
      if (c >= dv) break;
      float a = acc[i];
      for (int j = 0; j < FWD_BK; ++j) a += sP[row * (FWD_BK + 1) + j] * sV[j * sv_stride + c];
      acc[i] = a;
    }
  }
  lrow += __shfl_xor_sync(0xffffffffu, lrow, 1);
  lrow += __shfl_xor_sync(0xffffffffu, lrow, 2);
  const int qi = qs + row;
  if (qi < lq) {
    const float inv = lrow > 0.f ? 1.f / lrow : 0.f;
    const long long orow = elem_off(L.o, q0 + qi, h);
    for (int i = 0; i < ncol; ++i) {
      const int c = sub + 4 * i;
      if (c < dv) O[orow + c] = TypeOps<T>::from_f(acc[i] * inv);
    }
    if (sub == 0) {
      const long long li = group ? (long long)h * p.total_q + q0 + qi
                                 : ((long long)b * p.nhead_q + h) * p.seqlen_q + qi;
      p.lse[li] = lrow > 0.f ? (mrow + log2f(lrow)) * 0.6931471805599453f : -INFINITY;
    }
  }
}

size_t fwd_smem_bytes(int dqk, int dv) {
  return sizeof(float) * ((size_t)FWD_BQ * (dqk + 1) + (size_t)FWD_BK * (dqk + 1) +
                          (size_t)FWD_BK * dv + (size_t)FWD_BQ * (FWD_BK + 1));
}

template <typename T, int NC>
static void launch_fwd_typed(const attn_fwd_params& p, const FwdLayout& L, dim3 grid, size_t smem, int group,
                             cudaStream_t st) {
  cudaFuncSetAttribute(fwd_kernel<T, NC>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  fwd_kernel<T, NC><<<grid, FWD_THREADS, smem, st>>>(p, L, group);
}

template <typename T>
static void launch_fwd_dtype(const attn_fwd_params& p, const FwdLayout& L, dim3 grid, size_t smem, int group,
                             cudaStream_t st) {
  if (p.d_v > 128) launch_fwd_typed<T, 64>(p, L, grid, smem, group, st);
  else launch_fwd_typed<T, 32>(p, L, grid, smem, group, st);
}

void launch_fwd(const attn_fwd_params& p, const FwdLayout& L, cudaStream_t st) {
  const int group = p.cu_seqlens_q != nullptr;
  dim3 grid(cdiv(p.seqlen_q, FWD_BQ), p.nhead_q, p.batch);
  const size_t smem = fwd_smem_bytes(p.d_qk, p.d_v);
  switch (p.dtype) {
    case ATTN_BF16: launch_fwd_dtype<__nv_bfloat16>(p, L, grid, smem, group, st); break;
    case ATTN_FP16: launch_fwd_dtype<__half>(p, L, grid, smem, group, st); break;
    default: launch_fwd_dtype<float>(p, L, grid, smem, group, st); break;
  }
}

// Forward with no keys at all: every query row sees nothing, so O = 0 and
// LSE = -inf, the values of a fully masked row.  O rows are (row, head)
// vectors of whole 4-byte words at word boundaries; LSE is dense.
__global__ void __launch_bounds__(256) fwd_no_keys_kernel(attn_fwd_params p, Strides so, long long rows) {
  const int esize = p.dtype == ATTN_FP32 ? 4 : 2;
  const int wpv = p.d_v * esize / 4;
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long i0 = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  uint32_t* o = static_cast<uint32_t*>(p.o);
  const long long n = rows * p.nhead_q * wpv;
  for (long long i = i0; i < n; i += stride) {
    const long long rr = i / ((long long)p.nhead_q * wpv);
    const int rem = (int)(i - rr * p.nhead_q * wpv), hh = rem / wpv, wd = rem - hh * wpv;
    o[elem_off(so, rr, hh) * esize / 4 + wd] = 0u;
  }
  for (long long i = i0; i < rows * p.nhead_q; i += stride) p.lse[i] = -INFINITY;
}

void launch_fwd_no_keys(const attn_fwd_params& p, const FwdLayout& L, cudaStream_t st) {
  const long long rows = p.cu_seqlens_q != nullptr ? (long long)p.total_q : (long long)p.batch * p.seqlen_q;
  if (rows > 0) fwd_no_keys_kernel<<<256, 256, 0, st>>>(p, L.o, rows);
}

// ------------------------------------------------------------- SIMT backward
// One block per work item (segment, kv head, KV tile of BN keys); thread r
// owns key row r: it forms row r of S^T, P^T, dP^T, dS^T for each query tile
// and accumulates rows r of dK and dV in shared memory.  dQ partials of the
// tile are reduced over the block's keys and stored into the item's dq_acc
// slice (deterministic) or added atomically (single slice).

template <typename T>
__global__ void __launch_bounds__(BN) bwd_simt_kernel(Problem P) {
  extern __shared__ float smem[];
  const int item = blockIdx.x;
  if (item >= P.hdr[HDR_NITEMS]) return;
  const int4 it = P.items[item];
  const int b = it.x, hk = it.y, kt = it.z;
  const Seg sg = segment(P, b);
  const int dqk = P.dqk, dv = P.dv;
  const int ks = dqk + 1, vs = dv + 1;
  float* sK = smem;                     // [BN][dqk+1]
  float* sV = sK + BN * ks;             // [BN][dv+1]
  float* sdK = sV + BN * vs;            // [BN][dqk+1]
  float* sdV = sdK + BN * ks;           // [BN][dv+1]
  float* sQ = sdV + BN * vs;            // [BM][dqk]
  float* sdO = sQ + BM * dqk;           // [BM][dv]
  float* sdS = sdO + BM * dv;           // [BN][BM+1]
  float* sL = sdS + BN * (BM + 1);      // [BM] -LSE * log2(e)
  float* sD = sL + BM;                  // [BM]

  const T* Qg = static_cast<const T*>(P.q);
  const T* Kg = static_cast<const T*>(P.k);
  const T* Vg = static_cast<const T*>(P.v);
  const T* dOg = static_cast<const T*>(P.dout);
  const int r = threadIdx.x;
  const int kv0 = kt * BN;
  const int klen = min(BN, sg.lk - kv0);
  for (int i = r; i < BN * dqk; i += BN) {
    const int rr = i / dqk, c = i % dqk;
    sK[rr * ks + c] = rr < klen ? TypeOps<T>::to_f(Kg[elem_off(P.sk_, sg.k0 + kv0 + rr, hk) + c]) : 0.f;
    sdK[rr * ks + c] = 0.f;
  }
  for (int i = r; i < BN * dv; i += BN) {
    const int rr = i / dv, c = i % dv;
    sV[rr * vs + c] = rr < klen ? TypeOps<T>::to_f(Vg[elem_off(P.sv_, sg.k0 + kv0 + rr, hk) + c]) : 0.f;
    sdV[rr * vs + c] = 0.f;
  }
  const MaskArgs m = mask_args(P.mask, P.left, P.right, sg.lq, sg.lk);
  int qlo, qhi;
  qtile_range(m, sg.lq, sg.lk, kt, qlo, qhi);
  for (int h = hk * P.g; h < (hk + 1) * P.g; ++h) {
    for (int qt = qlo; qt < qhi; ++qt) {
      const int qs = qt * BM;
      __syncthreads();
      for (int i = r; i < BM * dqk; i += BN) {
        const int c = i / dqk, e = i % dqk;
        sQ[i] = qs + c < sg.lq ? TypeOps<T>::to_f(Qg[elem_off(P.sq_, sg.q0 + qs + c, h) + e]) : 0.f;
      }
      for (int i = r; i < BM * dv; i += BN) {
        const int c = i / dv, e = i % dv;
        sdO[i] = qs + c < sg.lq ? TypeOps<T>::to_f(dOg[elem_off(P.sdo_, sg.q0 + qs + c, h) + e]) : 0.f;
      }
      if (r < BM) {
        const bool ok = qs + r < sg.lq;
        const long long li = ok ? lse_row(P, b, h, sg, qs + r) : 0;
        sL[r] = ok ? P.nlse2[li] : -INFINITY;
        sD[r] = ok ? P.dvec[li] : 0.f;
      }
      __syncthreads();
      for (int c = 0; c < BM; ++c) {
        const int qi = qs + c, kk = kv0 + r;
        float s = 0.f, dp = 0.f;
        for (int e = 0; e < dqk; ++e) s += sK[r * ks + e] * sQ[c * dqk + e];
        for (int e = 0; e < dv; ++e) dp += sV[r * vs + e] * sdO[c * dv + e];
        const bool ok = r < klen && qi < sg.lq && visible(m, qi, kk);
        const float pr = ok ? fast_exp2(fmaf(s, P.scale_log2, sL[c])) : 0.f;
        const float ds = pr * (dp - sD[c]);
        sdS[r * (BM + 1) + c] = ds;
        for (int e = 0; e < dv; ++e) sdV[r * vs + e] += pr * sdO[c * dv + e];
        for (int e = 0; e < dqk; ++e) sdK[r * ks + e] += ds * sQ[c * dqk + e];
      }
      __syncthreads();
      for (int o = r; o < BM * dqk; o += BN) {
        const int c = o / dqk, e = o % dqk;
        if (qs + c >= sg.lq) continue;
        float a = 0.f;
        for (int rr = 0; rr < BN; ++rr) a += sdS[rr * (BM + 1) + c] * sK[rr * ks + e];
        const int tix = qtile_index(P, b, qt);
        if (!ATTN_INDEX_OK(P, tix >= 0 && tix < P.ntiles && (!P.det || kt < P.nsplits), 11)) continue;
        float* tile = dq_tile(P, P.det ? kt : 0, h, tix);
        if (P.det) tile[c * dqk + e] = a;
        else atomicAdd(tile + c * dqk + e, a);
      }
    }
  }
  __syncthreads();
  const int krow = sg.k0 + kv0 + r;
  if (r < klen && ATTN_INDEX_OK(P, krow >= 0 && krow < rows_k(P), 12)) {
    T* dK = static_cast<T*>(P.dk) + elem_off(P.sdk_, krow, hk);
    T* dV = static_cast<T*>(P.dv_out) + elem_off(P.sdv_, krow, hk);
    for (int e = 0; e < dqk; ++e) dK[e] = TypeOps<T>::from_f(sdK[r * ks + e] * P.scale);
    for (int e = 0; e < dv; ++e) dV[e] = TypeOps<T>::from_f(sdV[r * vs + e]);
  }
}

size_t bwd_simt_smem_bytes(int dqk, int dv) {
  return sizeof(float) * ((size_t)BN * (dqk + 1) * 2 + (size_t)BN * (dv + 1) * 2 + (size_t)BM * dqk +
                          (size_t)BM * dv + (size_t)BN * (BM + 1) + 2 * BM);
}

void launch_bwd_simt(const Problem& P, cudaStream_t st) {
  const size_t smem = bwd_simt_smem_bytes(P.dqk, P.dv);
  const int grid = P.max_items > 0 ? P.max_items : 1;
  switch (P.dtype) {
    case ATTN_BF16:
      cudaFuncSetAttribute(bwd_simt_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      bwd_simt_kernel<__nv_bfloat16><<<grid, BN, smem, st>>>(P);
      break;
    case ATTN_FP16:
      cudaFuncSetAttribute(bwd_simt_kernel<__half>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      bwd_simt_kernel<__half><<<grid, BN, smem, st>>>(P);
      break;
    default:
      cudaFuncSetAttribute(bwd_simt_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      bwd_simt_kernel<float><<<grid, BN, smem, st>>>(P);
      break;
  }
}

}  // namespace attn
