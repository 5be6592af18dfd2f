// Scheduler, preprocess and dQ reduce/convert kernels of the FMHA backward.
//
// * schedule: validates cu_seqlens on the device and writes the list of work
//   items (segment, kv head, KV tile) in KV-tile-major order, so the most
//   expensive causal tiles (lowest KV-tile index) are dealt first.  It replaces
//   the host-side seqstart copy CK's group-mode launcher needed (aiter PR
//   #2216 follow-up commit on the unified workspace: ".to(at::kCPU)").
// * preprocess: D = rowsum(dO * O) in fp32 and the log2-scaled LSE, plus the
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
  }
}

void launch_schedule(const Problem& P, cudaStream_t st) {
  schedule_kernel<<<1, 256, 0, st>>>(P);
}

// --------------------------------------------------------------- preprocess
// One warp per (packed token, query head): reads one O row and one dO row
// (d_v elements, contiguous) and writes D and the log2-scaled LSE.

template <typename T>
__global__ void __launch_bounds__(256) preprocess_kernel(Problem P, long long ntok) {
  const int lane = threadIdx.x & 31;
  const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  const T* O = static_cast<const T*>(P.o);
  const T* dO = static_cast<const T*>(P.dout);
  const float LOG2E = 1.4426950408889634f;
  for (long long r = warp; r < ntok * P.hq; r += nwarps) {
    const long long tok = r / P.hq;
    const int h = (int)(r - tok * P.hq);
    const T* orow = O + r * P.dv;
    const T* drow = dO + r * P.dv;
    float acc = 0.f;
    for (int c = lane; c < P.dv; c += 32)
      acc += TypeOps<T>::to_f(orow[c]) * TypeOps<T>::to_f(drow[c]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) {
      long long li;
      if (P.group) {
        li = (long long)h * P.tq + tok;
      } else {
        const long long b = tok / P.sq, q = tok - b * P.sq;
        li = (b * P.hq + h) * P.sq + q;
      }
      const float l = P.lse[li];
      P.dvec[li] = acc;
      P.lse2[li] = (l == -INFINITY) ? INFINITY : l * LOG2E;
    }
  }
  if (!P.det) {
    float4* acc4 = reinterpret_cast<float4*>(P.dq_acc);
    const long long n4 = P.n_lse * P.dqk / 4;
    const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long nt = (long long)gridDim.x * blockDim.x;
    for (long long i = t; i < n4; i += nt) acc4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
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
// One warp per (packed token, query head).  Deterministic mode sums, in
// ascending KV-tile order, exactly the slices whose KV tile reaches this
// row's query tile (the others were never written); atomic mode reads the
// single slice.

template <typename T>
__global__ void __launch_bounds__(256) reduce_convert_kernel(Problem P, long long ntok) {
  const int lane = threadIdx.x & 31;
  const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  T* dQ = static_cast<T*>(P.dq);
  const int nv = P.dqk / 4;
  const long long slice = P.n_lse * P.dqk;
  for (long long r = warp; r < ntok * P.hq; r += nwarps) {
    const long long tok = r / P.hq;
    const int h = (int)(r - tok * P.hq);
    int b, q;
    if (P.group) {
      // segment of this packed token: binary search of cu_seqlens_q
      int lo = 0, hi = P.nseg;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(P.cu_q + mid) <= tok) lo = mid; else hi = mid;
      }
      b = lo;
      q = (int)(tok - __ldg(P.cu_q + b));
    } else {
      b = (int)(tok / P.sq);
      q = (int)(tok - (long long)b * P.sq);
    }
    const Seg s = segment(P, b);
    const long long row = lse_row(P, b, h, s, q);
    const float* base = P.dq_acc + row * P.dqk;
    T* out = dQ + r * P.dqk;
    for (int v = lane; v < nv; v += 32) {
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
      if (P.det) {
        const MaskArgs m = mask_args(P.mask, P.left, P.right, s.lq, s.lk);
        const int qt = q / BM;
        int nkv = cdiv(s.lk, BN);
        if (nkv > P.nsplits) nkv = P.nsplits;   // guards cu_seqlens that broke their bound
        for (int kt = 0; kt < nkv; ++kt) {
          int lo, hi;
          qtile_range(m, s.lq, s.lk, kt, lo, hi);
          if (qt < lo || qt >= hi) continue;
          const float4 x = reinterpret_cast<const float4*>(base + (long long)kt * slice)[v];
          a.x += x.x; a.y += x.y; a.z += x.z; a.w += x.w;
        }
      } else if (s.lk > 0) {
        a = reinterpret_cast<const float4*>(base)[v];
      }
      out[4 * v + 0] = TypeOps<T>::from_f(a.x * P.scale);
      out[4 * v + 1] = TypeOps<T>::from_f(a.y * P.scale);
      out[4 * v + 2] = TypeOps<T>::from_f(a.z * P.scale);
      out[4 * v + 3] = TypeOps<T>::from_f(a.w * P.scale);
    }
  }
}

void launch_reduce_convert(const Problem& P, cudaStream_t st) {
  const long long ntok = P.group ? (long long)P.tq : (long long)P.nseg * P.sq;
  const int grid = num_sms() * 8;
  switch (P.dtype) {
    case ATTN_BF16: reduce_convert_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(P, ntok); break;
    case ATTN_FP16: reduce_convert_kernel<__half><<<grid, 256, 0, st>>>(P, ntok); break;
    default: reduce_convert_kernel<float><<<grid, 256, 0, st>>>(P, ntok); break;
  }
}

}  // namespace attn
