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

__global__ void __launch_bounds__(256) schedule_kernel(Problem P) {
  __shared__ int s_bad;
  const int tid = threadIdx.x;
  if (tid == 0) {
    s_bad = 0;
    P.hdr[HDR_STATUS] = 0;
    P.hdr[HDR_NEXT] = 0;
    P.hdr[HDR_DIAG] = 0;
  }
  if (tid >= 16 && tid < HDR_WORDS) P.hdr[tid] = 0;   // optional per-site wait counters
  __syncthreads();
  if (P.group) {
    for (int b = tid; b < P.nseg; b += blockDim.x) {
      const int q0 = P.cu_q[b], q1 = P.cu_q[b + 1];
      const int k0 = P.cu_k[b], k1 = P.cu_k[b + 1];
      bool bad = q1 < q0 || k1 < k0 || q1 - q0 > P.sq || k1 - k0 > P.sk;
      if (b == 0) bad |= q0 != 0 || k0 != 0;
      if (b == P.nseg - 1) bad |= q1 != P.tq || k1 != P.tk;
      if (bad) s_bad = 1;
    }
  }
  __syncthreads();
  if (s_bad) {
    if (tid == 0) {
      P.hdr[HDR_STATUS] = ATTN_ERR_BAD_SEQLENS;
      P.hdr[HDR_NITEMS] = 0;
    }
    return;
  }
  // KV-tile-major enumeration by warp 0: for kt, for segment, for kv head.
  if (tid < 32) {
    const int lane = tid;
    const int nkv_max = cdiv(P.sk > 0 ? P.sk : 1, BN);
    int n = 0;
    for (int kt = 0; kt < nkv_max; ++kt) {
      for (int b0 = 0; b0 < P.nseg; b0 += 32) {
        const int b = b0 + lane;
        bool has = false;
        if (b < P.nseg) {
          const int lk = P.group ? P.cu_k[b + 1] - P.cu_k[b] : P.sk;
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
      if (b < P.nseg) v = cdiv(P.cu_q[b + 1] - P.cu_q[b], BM);
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

void launch_schedule(const Problem& P, cudaStream_t st) {
  schedule_kernel<<<1, 256, 0, st>>>(P);
}

// --------------------------------------------------------------- preprocess
// D and -LSE*log2(e) of every (packed token, query head) row.  16-bit
// inputs: half a warp per row, 16-byte loads of O and dO.  fp32 inputs: one
// warp per row.  In atomic mode the single dq_acc slice is zeroed as well.

__device__ __forceinline__ void write_row_stats(const Problem& P, long long r, float acc) {
  const float LOG2E = 1.4426950408889634f;
  const long long tok = r / P.hq;
  const int h = (int)(r - tok * P.hq);
  long long li;
  if (P.group) {
    li = (long long)h * P.tq + tok;
  } else {
    const long long b = tok / P.sq, q = tok - b * P.sq;
    li = (b * P.hq + h) * P.sq + q;
  }
  const float l = P.lse[li];
  P.dvec[li] = acc;
  P.nlse2[li] = (l == -INFINITY) ? -INFINITY : -l * LOG2E;
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

template <typename T>
__global__ void __launch_bounds__(256) preprocess_kernel(Problem P, long long ntok) {
  const int lane = threadIdx.x & 31;
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long nthreads = (long long)gridDim.x * blockDim.x;
  const long long nrows = ntok * P.hq;
  if constexpr (sizeof(T) == 2) {
    // half warp per row; d_v is a multiple of 8 for the 16-bit kernels
    const int sub = lane & 15;
    const long long hw = tid >> 4, nhw = nthreads >> 4;
    const uint4* O = static_cast<const uint4*>(P.o);
    const uint4* dO = static_cast<const uint4*>(P.dout);
    const int nv = P.dv / 8;
    for (long long r0 = hw - (hw & 1); r0 < nrows; r0 += nhw) {
      const long long r = r0 + (hw & 1);
      float acc = 0.f;
      if (r < nrows)
        for (int v = sub; v < nv; v += 16) acc += dot8(O[r * nv + v], dO[r * nv + v], (T*)nullptr);
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (sub == 0 && r < nrows) write_row_stats(P, r, acc);
    }
  } else {
    const long long warp = tid >> 5, nwarps = nthreads >> 5;
    const T* O = static_cast<const T*>(P.o);
    const T* dO = static_cast<const T*>(P.dout);
    for (long long r = warp; r < nrows; r += nwarps) {
      float acc = 0.f;
      for (int c = lane; c < P.dv; c += 32)
        acc += TypeOps<T>::to_f(O[r * P.dv + c]) * TypeOps<T>::to_f(dO[r * P.dv + c]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) write_row_stats(P, r, acc);
    }
  }
  if (!P.det) {
    float4* acc4 = reinterpret_cast<float4*>(P.dq_acc);
    const long long n4 = (long long)P.hq * P.ntiles * P.dqk * BM / 4;
    for (long long i = tid; i < n4; i += nthreads) acc4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

static int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

void launch_preprocess(const Problem& P, cudaStream_t st) {
  const long long ntok = P.group ? (long long)P.tq : (long long)P.nseg * P.sq;
  const int grid = num_sms() * 8;
  switch (P.dtype) {
    case ATTN_BF16: preprocess_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(P, ntok); break;
    case ATTN_FP16: preprocess_kernel<__half><<<grid, 256, 0, st>>>(P, ntok); break;
    default: preprocess_kernel<float><<<grid, 256, 0, st>>>(P, ntok); break;
  }
}

// ----------------------------------------------------------- reduce/convert
// One block per (query head, query tile).  The dQ^T tiles of the slices whose
// KV tile reaches this query tile (the others were never written) are summed
// in ascending slice order; atomic mode reads the single slice.  The sum is
// transposed through shared memory, scaled and written as dQ rows.

constexpr int RC_THREADS = 256;

template <typename T>
__global__ void __launch_bounds__(RC_THREADS) reduce_convert_kernel(Problem P) {
  extern __shared__ float tile[];   // [dqk][BM + 1]
  const int dqk = P.dqk;
  const int nv4 = dqk * BM / 4;      // float4 per dQ^T tile
  const int ntq = cdiv(P.sq, BM);
  T* dQ = static_cast<T*>(P.dq);
  for (long long w = blockIdx.x; w < (long long)P.hq * P.ntiles; w += gridDim.x) {
    const int h = (int)(w / P.ntiles), t = (int)(w - (long long)h * P.ntiles);
    int b, qt;
    if (P.group) {
      if (t >= __ldg(P.tile_off + P.nseg)) continue;   // beyond the last segment's tiles
      int lo = 0, hi = P.nseg;                           // largest b with tile_off[b] <= t
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(P.tile_off + mid) <= t) lo = mid; else hi = mid;
      }
      b = lo;
      qt = t - __ldg(P.tile_off + b);
    } else {
      b = t / ntq;
      qt = t - b * ntq;
    }
    const Seg s = segment(P, b);
    const int nvalid = min(BM, s.lq - qt * BM);
    if (nvalid <= 0) continue;
    float4 acc[(192 * BM / 4 + RC_THREADS - 1) / RC_THREADS];
#pragma unroll
    for (int i = 0; i < (int)(sizeof(acc) / sizeof(acc[0])); ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    auto add_tile = [&](const float* src) {
      const float4* s4 = reinterpret_cast<const float4*>(src);
#pragma unroll
      for (int i = 0; i < (int)(sizeof(acc) / sizeof(acc[0])); ++i) {
        const int v = threadIdx.x + i * RC_THREADS;
        if (v < nv4) {
          const float4 x = __ldcs(s4 + v);
          acc[i].x += x.x; acc[i].y += x.y; acc[i].z += x.z; acc[i].w += x.w;
        }
      }
    };
    if (P.det) {
      const MaskArgs m = mask_args(P.mask, P.left, P.right, s.lq, s.lk);
      int nkv = cdiv(s.lk, BN);
      if (nkv > P.nsplits) nkv = P.nsplits;   // guards cu_seqlens that broke their bound
      for (int kt = 0; kt < nkv; ++kt) {
        int lo, hi;
        qtile_range(m, s.lq, s.lk, kt, lo, hi);
        if (qt >= lo && qt < hi) add_tile(dq_tile(P, kt, h, t));
      }
    } else if (s.lk > 0) {
      add_tile(dq_tile(P, 0, h, t));
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < (int)(sizeof(acc) / sizeof(acc[0])); ++i) {
      const int v = threadIdx.x + i * RC_THREADS;
      if (v < nv4) {
        if (P.det) {                 // query-major tiles: 4 consecutive d of one query
          const int c = (4 * v) / dqk, e = (4 * v) % dqk;
          float* dst = tile + e * (BM + 1) + c;
          dst[0] = acc[i].x; dst[BM + 1] = acc[i].y; dst[2 * (BM + 1)] = acc[i].z; dst[3 * (BM + 1)] = acc[i].w;
        } else {                     // d-major tile: 4 consecutive queries of one d
          const int e = (4 * v) / BM, c = (4 * v) % BM;
          float* dst = tile + e * (BM + 1) + c;
          dst[0] = acc[i].x; dst[1] = acc[i].y; dst[2] = acc[i].z; dst[3] = acc[i].w;
        }
      }
    }
    __syncthreads();
    const int nch = dqk / 8;                 // 8-element chunks per dQ row
    for (int u = threadIdx.x; u < nvalid * nch; u += RC_THREADS) {
      const int c = u / nch, ch = u - c * nch;
      T outv[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) outv[k] = TypeOps<T>::from_f(tile[(ch * 8 + k) * (BM + 1) + c] * P.scale);
      T* row = dQ + ((long long)(s.q0 + qt * BM + c) * P.hq + h) * dqk + ch * 8;
      if (sizeof(T) == 2) {
        *reinterpret_cast<uint4*>(row) = *reinterpret_cast<uint4*>(outv);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) row[k] = outv[k];
      }
    }
    __syncthreads();
  }
}

void launch_reduce_convert(const Problem& P, cudaStream_t st) {
  const long long work = (long long)P.hq * P.ntiles;
  if (work <= 0) return;
  const int grid = (int)(work < (long long)num_sms() * 16 ? work : (long long)num_sms() * 16);
  const size_t smem = (size_t)P.dqk * (BM + 1) * sizeof(float);
  switch (P.dtype) {
    case ATTN_BF16:
      cudaFuncSetAttribute(reduce_convert_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      reduce_convert_kernel<__nv_bfloat16><<<grid, RC_THREADS, smem, st>>>(P);
      break;
    case ATTN_FP16:
      cudaFuncSetAttribute(reduce_convert_kernel<__half>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      reduce_convert_kernel<__half><<<grid, RC_THREADS, smem, st>>>(P);
      break;
    default:
      cudaFuncSetAttribute(reduce_convert_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      reduce_convert_kernel<float><<<grid, RC_THREADS, smem, st>>>(P);
      break;
  }
}

}  // namespace attn
