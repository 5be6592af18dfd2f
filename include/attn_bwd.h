/*
 * attn_bwd.h - C ABI of the GB300 (sm_103a) fused multi-head attention
 * backward pass.
 *
 * Given Q, K, V, the forward output O, the upstream gradient dO and the
 * forward log-sum-exp LSE, attn_bwd computes dQ, dK and dV of softmax
 * attention.  The operation is the FMHA backward whose deterministic,
 * split-dQ persistent-kernel path is described in ROCm/aiter PR #2216
 * ("[CK_TILE] FMHA BWD Use Persistent Kernels in Deterministic Mode",
 * Motivation), behind a sizing call plus an execute call on one opaque
 * workspace as in that PR's follow-up commit "[CK_TILE] mha bwd: adapt to CK
 * #6152 unified workspace API".  Batch and group (THD, packed ragged) modes
 * follow ROCm/TransformerEngine PR #446 (the batch/group seqstart setup in
 * ck_fused_attn_bwd.cpp) and PR #671 (Summary, Root cause).
 *
 * Conventions
 * -----------
 * - Every pointer named "device" is a CUDA device pointer owned by the
 *   caller; the library allocates nothing and keeps no per-device state.
 * - All work is enqueued on the caller's stream; no call synchronises the
 *   host except attn_bwd_read_status and attn_bwd_timed.
 * - Return value: ATTN_OK (0) on success, a negative attn_status_t otherwise.
 *   Arguments are validated before anything is launched; an unsupported or
 *   inconsistent configuration is rejected, never computed silently
 *   (aiter PR #2216 follow-up: "LOG_ERROR + return -1" on missing group
 *   pointers; TransformerEngine PR #671: a hard head-dim check instead of a
 *   silent hard-coded size).
 * - Tensors are contiguous by default (per-tensor strides: see the stride_*
 *   fields of attn_bwd_params).  Batch mode (cu_seqlens_q == cu_seqlens_k ==
 *   NULL): q [B,Sq,Hq,d_qk], k [B,Sk,Hkv,d_qk], v [B,Sk,Hkv,d_v],
 *   o/dout/dq [B,Sq,Hq,·], dk/dv like k/v, lse [B,Hq,Sq].  Group mode:
 *   q [Tq,Hq,d_qk], k [Tk,Hkv,d_qk], v [Tk,Hkv,d_v], lse [Hq,Tq]; segment b
 *   owns rows cu_seqlens_q[b]..cu_seqlens_q[b+1] and keys
 *   cu_seqlens_k[b]..cu_seqlens_k[b+1] and attends only within itself.
 * - Padded group mode (cu_seqlens_q_padded / cu_seqlens_k_padded set): the
 *   logical length of segment b still comes from cu_seqlens (Lq_b =
 *   cu_seqlens_q[b+1] - cu_seqlens_q[b]), but its rows start at the
 *   physical row cu_seqlens_q_padded[b], so segment b owns rows
 *   padded[b] .. padded[b] + Lq_b - 1 and the rows up to padded[b+1] are
 *   padding (the seqstart convention of TransformerEngine PR #446, review of
 *   ck_fused_attn_fwd.cpp / ck_fused_attn_bwd.cpp, and of the "physical
 *   seqstart" in aiter PR #2216's unified-workspace follow-up commit).
 *   total_q / total_k then count physical rows, and lse is [Hq, total_q]
 *   indexed by physical row.  Rows that belong to no segment are written
 *   zero in dq, dk and dv.  Values in padding rows never reach a result,
 *   but those of q, k, v and dout must be finite (tiles that overlap padding
 *   multiply them by exact zeros).  Either side may be padded alone.
 * - Query head h reads kv head h / (Hq / Hkv) (GQA, contiguous groups).
 * - LSE is the natural-log log-sum-exp of the scaled scores, fp32; -inf
 *   marks a row with no visible key (its gradients are zero).
 */
#ifndef ATTN_BWD_H_
#define ATTN_BWD_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = -1,         /* null pointer, bad size, bad enum, misaligned */
  ATTN_ERR_UNSUPPORTED_HEADDIM = -2, /* (d_qk, d_v) not built for this dtype       */
  ATTN_ERR_WORKSPACE_TOO_SMALL = -3, /* workspace_bytes < attn_bwd_workspace_size   */
  ATTN_ERR_CUDA = -4,                /* a CUDA runtime/driver call failed           */
  ATTN_ERR_DEVICE_FLAG = -5,         /* kernels reported an error (see read_status) */
  ATTN_ERR_TIMEOUT = -6,             /* a bounded in-kernel wait expired            */
  ATTN_ERR_BAD_SEQLENS = -7          /* cu_seqlens (or the padded starts) not
                                        monotone, overlapping or beyond the bounds */
} attn_status_t;

/* Mask kinds: the AITER mask enum reviewed in TransformerEngine PR #446
 * (ck_to_aiter_mask_type).  With off = 0 for TOP_LEFT and off = Lk - Lq for
 * BOTTOM_RIGHT and WINDOW (per segment), key j is visible to query i iff
 *   CAUSAL_*: j <= i + off
 *   WINDOW:   i + off - window_left <= j <= i + off + window_right
 * (inclusive; -1 means unbounded on that side, other negative bounds are
 * rejected). */
typedef enum {
  ATTN_MASK_NONE = 0,
  ATTN_MASK_CAUSAL_TOP_LEFT = 1,
  ATTN_MASK_CAUSAL_BOTTOM_RIGHT = 2,
  ATTN_MASK_WINDOW = 3
} attn_mask_t;

/* Element type of q, k, v, o, dout, dq, dk, dv (lse is always fp32).
 * Supported head dims: BF16/FP16 (d_qk, d_v) in {(64,64), (128,128),
 * (192,128), (256,256)} on the tensor-core kernel (at (256,256) each KV tile
 * is processed in two passes over its query tiles, one per 128-column half of
 * dK, dV and dQ); FP32 d_qk in [4, 64] with d_qk % 4 == 0 and d_v in [1, 64]
 * on the fp32 SIMT kernel.  Any other pair returns
 * ATTN_ERR_UNSUPPORTED_HEADDIM before a launch (the loud head-dim check asked
 * for in the review of TE PR #671). */
typedef enum { ATTN_BF16 = 0, ATTN_FP16 = 1, ATTN_FP32 = 2 } attn_dtype_t;

/* Attention bias shapes: the bias of shape (bias_b, bias_h, s_q, s_kv) of
 * TransformerEngine PR #446 (review of ck_fused_attn_bwd.cpp, BiasShape
 * k11SS / k1HSS / kBHSS / kB1SS), contiguous with row stride seqlen_k, in the
 * dtype of q; bias_h counts query heads.  It is added to the scaled scores,
 * S = softmax_scale * Q K^T + bias, before the mask.  Batch mode and the
 * 16-bit dtypes only. */
typedef enum {
  ATTN_BIAS_NONE = 0,
  ATTN_BIAS_11SS = 1,   /* [1, 1, Sq, Sk]: one matrix for every batch entry and head */
  ATTN_BIAS_1HSS = 2,   /* [1, Hq, Sq, Sk] */
  ATTN_BIAS_BHSS = 3,   /* [B, Hq, Sq, Sk] */
  ATTN_BIAS_B1SS = 4    /* [B, 1, Sq, Sk] */
} attn_bias_t;

typedef struct {
  int32_t dtype;          /* attn_dtype_t                                          */
  int32_t batch;          /* batch mode: B; group mode: number of segments         */
  int32_t nhead_q;        /* Hq                                                    */
  int32_t nhead_kv;       /* Hkv, Hq % Hkv == 0                                    */
  int32_t seqlen_q;       /* batch: Sq; group: upper bound on every query segment  */
  int32_t seqlen_k;       /* batch: Sk; group: upper bound on every key segment    */
  int32_t total_q;        /* group mode: Tq = cu_seqlens_q[batch]; ignored in batch */
  int32_t total_k;        /* group mode: Tk = cu_seqlens_k[batch]; ignored in batch */
  int32_t d_qk;           /* head dim of q and k                                   */
  int32_t d_v;            /* head dim of v and o                                   */
  const int32_t* cu_seqlens_q; /* device, [batch+1], 4-byte aligned, or NULL
                                  (batch mode)                                  */
  const int32_t* cu_seqlens_k; /* device, [batch+1], 4-byte aligned, or NULL      */
  const int32_t* cu_seqlens_q_padded; /* device, [batch+1]: physical start row of
                             each query segment, or NULL (start = cu_seqlens_q);
                             group mode only.  Must satisfy padded[b] + Lq_b <=
                             padded[b+1] and padded[batch] <= total_q       */
  const int32_t* cu_seqlens_k_padded; /* same for keys and total_k            */
  int32_t mask;           /* attn_mask_t                                           */
  int32_t window_left;    /* ATTN_MASK_WINDOW only; -1 = unbounded                 */
  int32_t window_right;   /* ATTN_MASK_WINDOW only; -1 = unbounded                 */
  float softmax_scale;    /* s in S = s * Q K^T                                    */
  int32_t deterministic;  /* attn_det_t: 0 fp32 atomics; 1 and 2 bitwise
                             repeatable fixed-order dQ reduction              */
  const void* q;          /* device inputs, layouts above                          */
  const void* k;
  const void* v;
  const void* o;
  const void* dout;
  const float* lse;       /* device, fp32 natural log, 4-byte aligned              */
  void* dq;               /* device outputs, same dtype as q; fully overwritten.
                             q .. dv are 16-byte aligned (4-byte for FP32)     */
  void* dk;
  void* dv;
  /* Element strides {batch, row, head} of each tensor (the strided layouts of
   * the pages' stride_s_q / nhead_stride arguments, TransformerEngine PR #446,
   * ck_fused_attn_bwd.cpp); the head dimension itself is contiguous.  Batch
   * mode: element (b, s, h, c) is at b*stride[0] + s*stride[1] + h*stride[2]
   * + c.  Group mode: (t, h, c) at t*stride[1] + h*stride[2] + c; stride[0]
   * is ignored.  All three zero = the contiguous layout above, so a
   * zero-initialised struct keeps the contiguous convention.  Otherwise the
   * row and head strides must be positive (the batch stride too when
   * batch > 1) and, for BF16/FP16, multiples of 8 elements (16 bytes: the
   * tensor-memory-access and vector alignment).  With batch > 1 the batch
   * entries must follow each other either along rows (batch stride = seqlen
   * x row stride, as in BSHD or packed QKV) or along heads (batch stride =
   * nhead x head stride, as in BHSD or SBHD), the same way for every tensor
   * of the call; any other layout returns ATTN_ERR_INVALID_ARG.  Outputs
   * must not overlap one another or the inputs.  lse keeps its contiguous
   * layout. */
  int64_t stride_q[3];
  int64_t stride_k[3];
  int64_t stride_v[3];
  int64_t stride_o[3];
  int64_t stride_dout[3];
  int64_t stride_dq[3];
  int64_t stride_dk[3];
  int64_t stride_dv[3];
  /* Attention bias and dropout (TE PR #446: the bias shapes above; dropout
   * driven by the philox seed / offset pointers passed to ck_attn_bwd).  A
   * zero-initialised tail means neither. */
  int32_t bias_type;      /* attn_bias_t                                           */
  float dropout_p;        /* probability of dropping an attention weight, in
                             [0, 1); 0 = no dropout.  16-bit dtypes only       */
  const void* bias;       /* device, attn_bias_t shape, dtype of q, 2-byte aligned */
  void* dbias;            /* device output [B, Hq, Sq, Sk] in the dtype of q, the
                             gradient of the biased scores (dS), or NULL; needs a
                             bias.  Fully overwritten (zero where masked).  The
                             gradient of a broadcast bias is its sum over the
                             broadcast dimensions, left to the caller (the
                             pages' CK kernels also emit dbias in BHSS only)  */
  const uint64_t* philox_seed;   /* device, 8-byte aligned; read when dropout_p > 0 */
  const uint64_t* philox_offset; /* device, 8-byte aligned.  Weight (i, j) of
                             (batch or segment b, query head h) is kept when
                             word (i mod 4) of Philox4x32-10 with key (seed mod
                             2^32, seed div 2^32) and counter (lo32(n), j,
                             b * Hq + h, hi32(n)), n = offset + i div 4, is at
                             least floor(dropout_p * 2^32); kept weights are
                             scaled by 1 / (1 - dropout_p).  O must come from a
                             forward with the same mask (attn_fwd with the same
                             seed, offset and dropout_p)                     */
} attn_bwd_params;

/* Forward helper that produces O and LSE for benchmark and test inputs
 * (the forward pass implied by TransformerEngine PR #446's ck_attn_fwd).
 * Same field meanings and alignment rules as attn_bwd_params (q, k, v, o
 * 16-byte aligned, 4-byte for FP32; lse 4-byte aligned); o and lse are
 * outputs. */
typedef struct {
  int32_t dtype;
  int32_t batch;
  int32_t nhead_q;
  int32_t nhead_kv;
  int32_t seqlen_q;
  int32_t seqlen_k;
  int32_t total_q;
  int32_t total_k;
  int32_t d_qk;
  int32_t d_v;
  const int32_t* cu_seqlens_q;
  const int32_t* cu_seqlens_k;
  const int32_t* cu_seqlens_q_padded;
  const int32_t* cu_seqlens_k_padded;
  int32_t mask;
  int32_t window_left;
  int32_t window_right;
  float softmax_scale;
  const void* q;
  const void* k;
  const void* v;
  void* o;                /* device output [.., Hq, d_v], dtype; padding rows of a
                             padded group layout are left untouched            */
  float* lse;             /* device output, fp32 natural log (padding rows likewise) */
  int64_t stride_q[3];    /* element strides, as in attn_bwd_params             */
  int64_t stride_k[3];
  int64_t stride_v[3];
  int64_t stride_o[3];
  int32_t bias_type;      /* as in attn_bwd_params                                 */
  float dropout_p;
  const void* bias;
  const uint64_t* philox_seed;
  const uint64_t* philox_offset;
} attn_fwd_params;

/* dQ accumulation modes (attn_bwd_params.deterministic).  The per-KV-tile dQ
 * partials of one query tile are summed
 *   ATTN_DET_ATOMIC: with fp32 atomics in arrival order (not repeatable);
 *   ATTN_DET_ORDERED: in ascending KV-tile order, each partial added into one
 *     fp32 dq_acc tile in turn (a per-tile turn counter serialises the adds,
 *     so the sum is bitwise repeatable; partials never leave the L2 cache
 *     as separate slices; at head dim 256 each column half has its own
 *     counters).  FP32 inputs use the split slices instead;
 *   ATTN_DET_SPLIT: each partial stored to its own dq_acc slice, nsplits =
 *     ceil(seqlen_k / 128), then summed in ascending slice order by a
 *     reduction kernel -- the split workspace of aiter PR #2216 (Motivation).
 * ORDERED and SPLIT perform the same fp32 additions in the same order and
 * give the same bits, except that ORDERED flushes subnormal partial sums to
 * zero (fp32 global reductions do). */
typedef enum { ATTN_DET_ATOMIC = 0, ATTN_DET_ORDERED = 1, ATTN_DET_SPLIT = 2 } attn_det_t;

/* Workspace bytes attn_bwd needs for *p.  Pure host arithmetic on the scalar
 * fields (no device access, no GPU probe), using the same layout function as
 * attn_bwd, so the sizing and the launch cannot disagree (the sizing-pass
 * lesson of TransformerEngine PR #671, review reply on is_v3_api_check).
 * The workspace is dominated by fp32 dq_acc slices, each Hq x ntiles query
 * tiles of 64 rows x d_qk, with ntiles = batch * ceil(seqlen_q / 64) in batch
 * mode and min(floor(total_q / 64) + batch, batch * ceil(seqlen_q / 64)) in
 * group mode (each segment's rows start a new tile: a per-segment padded
 * layout, the kind TransformerEngine PR #671's Fix switches dq_acc to, with
 * one layout shared by the sizing call and the kernels).  ATTN_DET_SPLIT (and
 * ATTN_DET_ORDERED with FP32 inputs) uses nsplits = ceil(seqlen_k / 128)
 * slices, the other modes one; ATTN_DET_ORDERED adds a turn counter per
 * query tile and head (two at d_qk = 256, one per column half).  Small per-row and per-tile tables come on top.
 * Writes the size to *bytes.  Returns ATTN_OK or an error code. */
int attn_bwd_workspace_size(const attn_bwd_params* p, size_t* bytes);

/* Enqueue the backward pass on `stream`.  `workspace` is a device buffer of
 * at least attn_bwd_workspace_size bytes, 256-byte aligned; its contents on
 * entry are irrelevant (the library initialises what it needs) and it must
 * not be used by another attn_bwd call in flight.  dq, dk, dv are fully
 * overwritten.  A problem with no query rows or no key rows in total (batch
 * x seqlen, or total_q / total_k in group mode, equal to 0) runs no attention
 * kernel: the other side's gradients are zeroed (no keys: every row sees
 * nothing, dQ = 0; no queries: dK = dV = 0), the tensors of the empty side
 * may be null and cu_seqlens are not read.  Invalid arguments return an
 * error before any launch;
 * problems found on the device (cu_seqlens inconsistent with the declared
 * bounds, an expired wait) are recorded in the workspace and returned by
 * attn_bwd_read_status. */
int attn_bwd(const attn_bwd_params* p, void* workspace, size_t workspace_bytes,
             cudaStream_t stream);

/* attn_bwd plus CUDA-event timing of its stages; synchronises `stream`
 * before returning.  stage_ms[0] = schedule + preprocess, [1] = main kernel,
 * [2] = dQ reduce/convert, [3] = the whole call. */
int attn_bwd_timed(const attn_bwd_params* p, void* workspace, size_t workspace_bytes,
                   cudaStream_t stream, float stage_ms[4]);

/* Synchronise `stream` and return the device status word of the last
 * attn_bwd run on `workspace` (ATTN_OK or an attn_status_t) in *status. */
int attn_bwd_read_status(const void* workspace, cudaStream_t stream, int* status);

/* Enqueue the forward helper on `stream`.  With no key rows in total every
 * query row sees nothing: O = 0 and LSE = -inf, the values of a fully masked
 * row; with no query rows nothing is written.  The tensors of an empty side
 * may be null. */
int attn_fwd(const attn_fwd_params* p, cudaStream_t stream);

/* Static description of a status code. */
const char* attn_status_string(int status);

/* Host-side tensors of attn_bwd_host: page-locked (pinned) host memory in
 * the contiguous layouts above.  q, k, v, o, dout, lse are read; dq, dk, dv
 * are written. */
typedef struct {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const void* dout;
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
} attn_host_tensors;

/* attn_bwd for inputs and outputs in host memory: copies Q, K, V, O, dO and
 * LSE from `host` into the device buffers of *p, runs the backward pass and
 * copies dQ, dK, dV back into `host`.  *p is an ordinary attn_bwd problem whose
 * tensor pointers are the caller's contiguous device staging buffers (all
 * strides zero).  The problem is split into at most `chunks` (1..64) parts:
 * runs of consecutive batch entries while chunks <= batch, else single
 * entries (group mode: the whole packed tensor) times runs of kv heads with
 * their query heads, whose head slices travel as 2-D copies (one line per
 * row; on a GB300 these run far below the plain copies' ~200 GB/s, so
 * chunks <= batch is the fast choice).  Chunk c's inputs are copied on
 * `copy_in` (O, dO and LSE first, so that its preprocess overlaps the copies
 * of Q, K and V), its backward runs on `stream`, its gradients are copied on
 * `copy_out` (dK and dV once the main kernel is done, during the dQ
 * conversion, then dQ), so one chunk's copies overlap another chunk's
 * compute.  The three streams must be distinct; the copies
 * start after the work already queued on `stream`, and `stream` completes
 * only once the last gradients are in host memory (synchronise it before
 * reading them).  Each chunk runs the same kernels in the same order as
 * attn_bwd, so the deterministic modes give the same bits as one attn_bwd
 * call.  The workspace is sized by attn_bwd_workspace_size(p) and reused by
 * the chunks in turn; a device-side failure in one chunk is kept in it (read
 * with attn_bwd_read_status) and the later chunks skip their work.  Returns
 * ATTN_OK when everything was enqueued, an error code otherwise. */
int attn_bwd_host(const attn_bwd_params* p, const attn_host_tensors* host, void* workspace,
                  size_t workspace_bytes, cudaStream_t stream, cudaStream_t copy_in, cudaStream_t copy_out,
                  int chunks);

/* Size of the device array attn_bwd_static_ws uses as its workspace. */
#define ATTN_BWD_STATIC_WS_BYTES (64u << 20)

/* attn_bwd for callers that cannot allocate device memory (for example code
 * that runs where cudaMalloc is forbidden or whose allocator is not reachable
 * from the call site).  The cited PRs have no counterpart: it is an addition
 * of this library.  The caller still passes every input and output through *p;
 * the workspace is a fixed ATTN_BWD_STATIC_WS_BYTES device array inside the
 * library (held on every GPU that loads the library until the process
 * exits), so no memory is allocated by this call.
 * - Problems whose attn_bwd_workspace_size exceeds ATTN_BWD_STATIC_WS_BYTES
 *   are rejected with ATTN_ERR_WORKSPACE_TOO_SMALL before anything runs.
 * - The first call while a given device is current looks up the array's
 *   device address (cudaGetSymbolAddress); make that first call before any
 *   stream capture on that device.
 * - That address is kept per device ordinal for the life of the process and
 *   belongs to the device's primary context.  After cudaDeviceReset, or with
 *   a non-primary context current, it no longer names the library's array:
 *   neither case is supported by this entry point (use attn_bwd there).
 * - All calls on a device share the one array: calls that overlap on the GPU
 *   (other streams, other host threads) race and corrupt each other.  Calls
 *   ordered on one stream are safe; each call initialises what it reads.
 * - Problems found on the device (cu_seqlens breaking their bounds) are
 *   recorded in the library's array, which this entry point does not expose;
 *   use attn_bwd with a caller workspace when that status is needed. */
int attn_bwd_static_ws(const attn_bwd_params* p, cudaStream_t stream);

/* Self-test of the bounded waits the backward kernels rely on (the pages ask
 * for loud failure instead of silent corruption: aiter PR #2216's launcher
 * returns an error, TE PR #671's check aborts).  One CTA runs, each bounded
 * at 1 ms:
 *   status[0]: an mbarrier wait whose phase never completes -> ATTN_ERR_TIMEOUT;
 *   status[1]: a wait for a turn counter that nobody advances -> ATTN_ERR_TIMEOUT;
 *   status[2]: the same wait entered after another CTA recorded an error,
 *              which must give up at once -> ATTN_OK when it did.
 * No GPU fault, trap or unbounded wait is involved.  `scratch` is a device
 * buffer of at least 3 * 128 * 4 + 16 bytes, 16-byte aligned, owned by the
 * caller; its contents are overwritten.  Synchronises `stream`.  Returns
 * ATTN_OK when the test ran (the results are in status), an error otherwise. */
int attn_selftest_waits(void* scratch, size_t scratch_bytes, cudaStream_t stream, int status[3]);

#ifdef __cplusplus
}
#endif
#endif /* ATTN_BWD_H_ */
