// The tensor-core backward kernel (tc_kernel.cuh) instantiated without the
// attention bias / dropout extras, the host entry that dispatches to it (and
// to the extras instantiations of tc_kernel_fx.cu), and the bounded-wait
// self-test.
#include "tc_kernel.cuh"

namespace attn {
namespace tc {

// ---------------------------------------------------------- wait self-test
// The bounded waits of the backward kernel, run on waits that can never end:
// an mbarrier whose phase nobody completes, a turn counter nobody advances,
// and a turn wait entered after another CTA has already failed.  Each gives up
// (within `limit_ns`, or at once in the last case) and records its status in
// its own header, as the backward kernel does; no fault, trap or hang.
constexpr uint64_t SELFTEST_LIMIT_NS = 1000000ull;   // 1 ms

__global__ void __launch_bounds__(32) selftest_waits_kernel(int* hdrs, uint32_t* counter) {
  constexpr uint64_t limit_ns = SELFTEST_LIMIT_NS;
  __shared__ __align__(8) uint64_t bar[1];
  __shared__ int abort_flag[3];
  if (threadIdx.x != 0) return;
  abort_flag[0] = abort_flag[1] = abort_flag[2] = 0;
  mbar_init(bar, 1);
  fence_mbar_init();
  const Ctx c0{bar, abort_flag + 0, hdrs};
  const Ctx c1{bar, abort_flag + 1, hdrs + HDR_WORDS};
  const Ctx c2{bar, abort_flag + 2, hdrs + 2 * HDR_WORDS};
  if (wait_bar<limit_ns>(c0, 0, 0, 42)) hdrs[HDR_DIAG] = -1;                 // must not succeed
  if (acquire_turn<limit_ns>(c1, counter, 1u)) hdrs[HDR_WORDS + HDR_DIAG] = -1;
  hdrs[2 * HDR_WORDS + HDR_STATUS] = ATTN_ERR_DEVICE_FLAG;          // "another CTA failed"
  const uint64_t t0 = globaltimer();
  const bool got = acquire_turn<limit_ns>(c2, counter, 1u);
  hdrs[2 * HDR_WORDS + HDR_DIAG] = (!got && globaltimer() - t0 < limit_ns / 2) ? 1 : 0;
}

int selftest_waits(void* scratch, size_t bytes, cudaStream_t st, int status[3]) {
  const size_t need = 3 * HDR_WORDS * sizeof(int) + 16;
  if (!scratch || bytes < need || (reinterpret_cast<uintptr_t>(scratch) & 15u) != 0) return ATTN_ERR_INVALID_ARG;
  int* hdrs = static_cast<int*>(scratch);
  uint32_t* counter = reinterpret_cast<uint32_t*>(hdrs + 3 * HDR_WORDS);
  if (cudaMemsetAsync(scratch, 0, need, st) != cudaSuccess) return ATTN_ERR_CUDA;
  selftest_waits_kernel<<<1, 32, 0, st>>>(hdrs, counter);
  int h[3 * HDR_WORDS];
  if (cudaMemcpyAsync(h, scratch, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess) return ATTN_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return ATTN_ERR_CUDA;
  status[0] = h[HDR_DIAG] == 42 ? h[HDR_STATUS] : ATTN_ERR_DEVICE_FLAG;
  status[1] = h[HDR_WORDS + HDR_DIAG] == 33 ? h[HDR_WORDS + HDR_STATUS] : ATTN_ERR_DEVICE_FLAG;
  status[2] = h[2 * HDR_WORDS + HDR_DIAG] == 1 ? ATTN_OK : ATTN_ERR_DEVICE_FLAG;
  return ATTN_OK;
}

}  // namespace tc

int launch_bwd_tc_fx(const Problem& P, cudaStream_t st);   // tc_kernel_fx.cu

int selftest_waits(void* scratch, size_t bytes, cudaStream_t st, int status[3]) {
  return tc::selftest_waits(scratch, bytes, st, status);
}

int launch_bwd_tc(const Problem& P, cudaStream_t st) {
  if (P.extras) return launch_bwd_tc_fx(P, st);
  if (P.dtype == ATTN_FP16) return tc::launch_mode<__half, false>(P, st);
  return tc::launch_mode<__nv_bfloat16, false>(P, st);
}

}  // namespace attn
