/*
 * spa.h -- C ABI of the GB300 (sm_103a) projected-feature softmax attention
 * library, libspa.so.
 *
 * The operation (per batch b and head h):
 *     Qp = Q P_h,  Kp = K P_h                P_h in R^{d x m}
 *     O  = softmax( Qp Kp^T / sqrt(m) ) V    row-wise softmax, full N x N
 * as defined by "Sparse Projection Attention: A Computationally Efficient
 * Framework for Long Sequence Modeling" (Sec. 3.1.2, Sec. 3.1.3, Algorithm 1)
 * and by steps 1-3 of Algorithm 2.1 of the "Projection-Decomposition
 * Attention" page (steps 4-5, the rank-r factorisation, are not part of this
 * library).  With causal != 0 query i only attends to keys j <= i (square,
 * top-left aligned mask).
 *
 * Conventions shared by every entry point
 *   Layout     all tensors dense, row-major, no padding:
 *                q, k   [B][H][N][d]      v, out  [B][H][N][d_v]
 *                P      [H][d][m]         one projection per head, shared by all b
 *   dtype      SPA_F32 or SPA_BF16; q, k, v and P all have this element type.
 *              Outputs are always fp32.
 *   Memory     unless an entry point says otherwise, every pointer is a CUDA
 *              device pointer on the current device, 16-byte aligned.  The
 *              caller owns every buffer it passes.  Between calls the library
 *              keeps, per device: a memory pool for the workspaces it takes
 *              itself (what it has reserved stays reserved until
 *              spa_host_pool_trim), the device error word, the internal
 *              streams of spa_attention_fwd_host, and the fixed scratch array
 *              of spa_attention_fwd_noalloc.
 *   stream     a cudaStream_t passed as void* (NULL = legacy default stream).
 *              Work is enqueued asynchronously; the return value reports
 *              argument errors and launch errors only.  Faults inside a kernel
 *              surface at the caller's next synchronisation.
 *   Empty      if B*H*N == 0 the call returns SPA_OK and touches nothing.
 *   Errors     a non-zero return is an spa_status; nothing was enqueued unless
 *              the status is SPA_ERR_CUDA from a launch.
 *   Threads    all entry points are reentrant.
 */
#ifndef SPA_H
#define SPA_H

#include <stddef.h>

/* Every entry point below is exported from libspa.so; the library is built
 * with hidden visibility, so nothing else is. */
#if defined(__GNUC__)
#define SPA_API __attribute__((visibility("default")))
#else
#define SPA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SPA_OK = 0,
  SPA_ERR_NULL = 1,        /* a required pointer is NULL                      */
  SPA_ERR_SHAPE = 2,       /* a size is negative or too large                 */
  SPA_ERR_DTYPE = 3,       /* dtype is not SPA_F32 / SPA_BF16                 */
  SPA_ERR_ALIGN = 4,       /* a pointer is not 16-byte aligned                */
  SPA_ERR_UNSUPPORTED = 5, /* shape outside what the kernels implement        */
  SPA_ERR_NOMEM = 6,       /* workspace allocation failed / too small         */
  SPA_ERR_CUDA = 7,        /* a CUDA runtime or driver call failed            */
  SPA_ERR_TIMEOUT = 8      /* a kernel gave up on a bounded wait (device word) */
} spa_status;

typedef enum { SPA_F32 = 0, SPA_BF16 = 1 } spa_dtype;

/* Human-readable name of a status code (static storage, never NULL). */
SPA_API const char *spa_status_str(int status);

/* Library ABI version: major * 10000 + minor * 100 + patch. */
SPA_API int spa_version(void);

/*
 * spa_project -- the projection step alone: x_proj[b][h][i][:] = x[b][h][i][:] P_h
 * (SPA Algorithm 1 steps 2-3; PDA Algorithm 2.1 step 1).
 *   x       [B][H][N][d] of `dtype`, device.
 *   P       [H][d][m] of `dtype`, device.
 *   x_proj  [B][H][N][m] fp32, device, written.
 * Products of the inputs are formed exactly and summed in fp32.
 * Supported: 1 <= d <= 256, 1 <= m <= 128.
 */
SPA_API int spa_project(const void *x, const void *P, float *x_proj, int B, int H, int N, int d,
                        int m, int dtype, void *stream);

/*
 * spa_attention_fwd -- the whole forward: projection, scores, (causal mask),
 * online softmax and the value product, without forming the N x N matrix.
 *   q, k    [B][H][N][d] of `dtype`, device.
 *   v       [B][H][N][d_v] of `dtype`, device.
 *   P       [H][d][m] of `dtype`, device.
 *   out     [B][H][N][d_v] fp32, device, written.
 *   causal  0 = full attention, non-zero = key j visible to query i iff j <= i.
 * Supported:
 *   SPA_BF16: 1 <= d <= 256; m in {16, 32, 64, 128}; d_v in {64, 128}.
 *   SPA_F32 : 1 <= d <= 256; 1 <= m <= 128;          1 <= d_v <= 256.
 *   N up to 2^31 - 1, B*H up to 65535.
 * Range (SPA_BF16): the softmax accumulates probabilities up to 2^40 times the
 * row's running maximum between rescales, so the output is finite for value
 * magnitudes |v| below 2^(87 - log2 N) (2^70 at N = 131072).
 * A workspace of spa_attention_workspace_size() bytes is taken on `stream`
 * from the memory pool the library keeps per device and given back to it on
 * the same stream (SPA_ERR_NOMEM if the allocation fails).  The pool keeps its
 * reservation across synchronisations, so a synchronised loop of calls does
 * not reserve device memory again; spa_host_pool_trim releases it.
 */
SPA_API int spa_attention_fwd(const void *q, const void *k, const void *v, const void *P,
                              float *out, int B, int H, int N, int d, int m, int d_v, int causal,
                              int dtype, void *stream);

/*
 * spa_attention_workspace_size -- bytes of device workspace the forward needs
 * for these sizes (0 when B*H*N == 0).  Validates like spa_attention_fwd.
 */
SPA_API int spa_attention_workspace_size(int B, int H, int N, int d, int m, int d_v, int dtype,
                                         size_t *bytes);

/*
 * spa_attention_fwd_ws -- spa_attention_fwd with a caller-provided workspace
 * (device, 256-byte aligned, at least spa_attention_workspace_size() bytes;
 * SPA_ERR_NOMEM if smaller).  The workspace is overwritten; it must not be in
 * use by other work on other streams while this call's kernels run.
 */
SPA_API int spa_attention_fwd_ws(const void *q, const void *k, const void *v, const void *P,
                                 float *out, int B, int H, int N, int d, int m, int d_v, int causal,
                                 int dtype, void *workspace, size_t workspace_bytes, void *stream);

/*
 * spa_attention_prepare / spa_attention_apply -- the forward in two stages on
 * a caller-provided workspace (as for spa_attention_fwd_ws).  prepare runs the
 * projection of q and k and leaves the score operands in the workspace; apply
 * runs scores, mask, online softmax and the value product from it.  The pair,
 * called in order on one stream with the same sizes, computes exactly what
 * spa_attention_fwd_ws computes.  apply may be repeated (other v, other
 * causal) on one prepared workspace as long as q, k, P and the sizes are
 * unchanged.  d_v must be passed to prepare as well: it takes part in the
 * size checks.
 */
SPA_API int spa_attention_prepare(const void *q, const void *k, const void *P, int B, int H, int N,
                                  int d, int m, int d_v, int dtype, void *workspace,
                                  size_t workspace_bytes, void *stream);
SPA_API int spa_attention_apply(const void *v, float *out, int B, int H, int N, int d, int m,
                                int d_v, int causal, int dtype, const void *workspace,
                                size_t workspace_bytes, void *stream);

/*
 * spa_attention_fwd_host -- end-to-end form on HOST buffers: copies q, k, v, P
 * to the device, runs the forward, copies out back, and synchronises `stream`
 * before returning, so `out` is valid on return.  Heads are independent, so
 * the (batch, head) range is cut into chunks of whole heads (at least about
 * 32 MB of traffic each, at most 32 chunks) that run on four internal
 * streams (created by the first call on a device and kept until the process
 * exits; concurrent calls share them) forked from and joined back into
 * `stream`: later chunks are copied
 * in and earlier ones copied out while a chunk computes.  The result is bit for
 * bit that of spa_attention_fwd.  Device buffers and workspace for four chunks
 * are taken on `stream` from a memory pool the library keeps per device and
 * released to it before return; the pool holds on to what it has reserved, so
 * that later calls do not reserve device memory again (spa_host_pool_trim
 * hands it back to the driver).
 * Page-locked host buffers give asynchronous, full-bandwidth copies; pageable
 * ones work but copy synchronously.  Same shapes and dtypes as
 * spa_attention_fwd.
 */
SPA_API int spa_attention_fwd_host(const void *q, const void *k, const void *v, const void *P,
                                   float *out, int B, int H, int N, int d, int m, int d_v,
                                   int causal, int dtype, void *stream);

/* spa_host_pool_trim -- releases the current device's unused memory kept by
 * the library's pool (the workspaces of the allocating entry points, the
 * staging of spa_attention_fwd_host, the scratch of spa_attention_decode; call
 * when none of them is running on that device). */
SPA_API int spa_host_pool_trim(void);

/*
 * spa_attention_fwd_noalloc -- spa_attention_fwd without any device
 * allocation.  (The pages describe no such entry point; it is an addition for
 * callers that cannot allocate device memory while they run -- code inside a
 * framework or allocator that owns all device memory, real-time loops that
 * must not enter the driver's allocator, processes with a fixed memory
 * budget.)  Same arguments, layouts and results as spa_attention_fwd.
 *   Scratch   a 64 MiB array compiled into libspa.so as device memory; every
 *             GPU that loads the library holds it until the process exits.
 *             Problems whose workspace (spa_attention_workspace_size) exceeds
 *             64 MiB are rejected with SPA_ERR_NOMEM before anything runs.
 *   Set-up    the first call on a device looks up the array's device address
 *             (cudaGetSymbolAddress) with that device current; make that first
 *             call before any stream capture.
 *   Sharing   all calls on a device share the one array.  Calls whose kernels
 *             overlap on the GPU (other streams, other threads) race on it:
 *             serialise them.  Contents left by an earlier call are never read.
 *   No cudaMalloc, cudaFree or other allocating routine is called.
 */
SPA_API int spa_attention_fwd_noalloc(const void *q, const void *k, const void *v, const void *P,
                                      float *out, int B, int H, int N, int d, int m, int d_v,
                                      int causal, int dtype, void *stream);

/*
 * spa_attention_fwd_lse -- spa_attention_fwd that also writes, for every query
 * row, the log-sum-exp of its logits (natural log):
 *   lse[b][h][i] = log sum_{j visible} exp(<Qp_i, Kp_j> / sqrt(m))
 * lse is [B][H][N] fp32, device, 4-byte aligned.  It is what
 * spa_attention_bwd_lse needs to recompute the probabilities A_ij =
 * exp(s_ij - lse_i) without a second forward.  Limits and workspace as
 * spa_attention_fwd.
 */
SPA_API int spa_attention_fwd_lse(const void *q, const void *k, const void *v, const void *P,
                                  float *out, float *lse, int B, int H, int N, int d, int m,
                                  int d_v, int causal, int dtype, void *stream);

/*
 * spa_attention_bwd -- gradients of spa_attention_fwd for an upstream gradient
 * dO [B][H][N][d_v] (same type as the inputs), given the forward's output out
 * (fp32).  Writes dq, dk [B][H][N][d], dv [B][H][N][d_v] and dP [H][d][m] (the
 * projection is shared by the batch: dP sums over it), all fp32:
 *   A = softmax(Qp Kp^T / sqrt(m)) (causal: keys j <= i), D_i = <dO_i, out_i>,
 *   dS = A * (dO V^T - D) / sqrt(m), dQp = dS Kp, dKp = dS^T Qp, dV = A^T dO,
 *   dq = dQp P_h^T, dk = dKp P_h^T, dP_h = sum_b (q^T dQp + k^T dKp)
 * ("Sparse Projection Attention", Sec. 3.4.1; Algorithm 2 trains P through
 * these).  d <= 128; the other limits are the forward's; every pointer 16-byte
 * aligned, else SPA_ERR_ALIGN.  Both implementations are flash-style: A and dS
 * are recomputed from the forward's row log-sum-exp and never stored.
 *   tensor cores (SPA_BF16, d in {64, 128}, m in {16, 32, 64}, d_v in
 *     {64, 128}): A and dS tile by tile in tensor memory.  The scores use the
 *     forward's own operands; P^T and dS are rounded to bf16 for their
 *     products (fp32 accumulation), dQp / dKp are carried into dq, dk, dP as
 *     bf16 hi + lo pairs (16 significant bits).
 *   CUDA cores (every other shape: SPA_F32, or m = 128, or another d):
 *     the same chain rule in fp32, one warp per key row (dV, dKp) and per
 *     query row (dQp).
 * spa_attention_bwd runs the forward once more for the log-sum-exp;
 * spa_attention_bwd_lse takes it.  Workspace on `stream` from the library's
 * pool (as for spa_attention_fwd).  An empty problem (B*H*N == 0) zeroes dP.
 */
SPA_API int spa_attention_bwd(const void *q, const void *k, const void *v, const void *P,
                              const float *out, const void *dO, float *dq, float *dk, float *dv,
                              float *dP, int B, int H, int N, int d, int m, int d_v, int causal,
                              int dtype, void *stream);
/* spa_attention_bwd_lse -- the same with the forward's lse ([B][H][N] fp32, as
 * written by spa_attention_fwd_lse; SPA_ERR_NULL if missing), so neither path
 * runs its own forward. */
SPA_API int spa_attention_bwd_lse(const void *q, const void *k, const void *v, const void *P,
                                  const float *out, const float *lse, const void *dO, float *dq,
                                  float *dk, float *dv, float *dP, int B, int H, int N, int d,
                                  int m, int d_v, int causal, int dtype, void *stream);

/*
 * The fused backward in three stages on a caller-provided workspace (device,
 * 256-byte aligned, at least spa_attention_bwd_workspace_size() bytes; the
 * stages must run in order on one stream with the same sizes and workspace).
 * Tensor-core shapes only (SPA_BF16, d in {64, 128}, m in {16, 32, 64}, d_v
 * in {64, 128}; otherwise SPA_ERR_UNSUPPORTED); pointers 16-byte aligned.
 *   prepare: the forward's score operands, bf16 Qp / Kp tiles, row statistics
 *            (D_i = <dO_i, out_i>, lse) and a zeroed dQp accumulator.
 *   apply:   the tensor-core kernel; writes dv and leaves dQp, dKp (fp32) in
 *            the workspace.
 *   finish:  dq, dk, dP from dQp, dKp in one tensor-core pass (dP is summed
 *            with floating-point reduce-adds whose order may vary).
 * prepare + apply + finish gives spa_attention_bwd_lse's dq, dk, dv bit for bit.
 */
SPA_API int spa_attention_bwd_workspace_size(int B, int H, int N, int d, int m, int d_v,
                                             int dtype, size_t *bytes);
SPA_API int spa_attention_bwd_prepare(const void *q, const void *k, const void *P,
                                      const float *out, const float *lse, const void *dO, int B,
                                      int H, int N, int d, int m, int d_v, int dtype,
                                      void *workspace, size_t workspace_bytes, void *stream);
SPA_API int spa_attention_bwd_apply(const void *v, const void *dO, float *dv, int B, int H, int N,
                                    int d, int m, int d_v, int causal, int dtype, void *workspace,
                                    size_t workspace_bytes, void *stream);
SPA_API int spa_attention_bwd_finish(const void *q, const void *k, const void *P, float *dq,
                                     float *dk, float *dP, int B, int H, int N, int d, int m,
                                     int d_v, int dtype, void *workspace, size_t workspace_bytes,
                                     void *stream);

/*
 * Decode with a projected key cache.  A decode step attends one new query per
 * (batch, head) to all cached keys; with the projection it needs the cached
 * K~ = K P_h (m values per key) instead of K (d values per key) ("Sparse
 * Projection Attention", Sec. 3.1.2; the cache saving is the pages' argument
 * for projected keys).  bf16 inputs only; d <= 256, m in {16,32,64,128}.
 *
 * Cache layout (caller-owned device memory, 16-byte aligned):
 *   kc      [B][H][cap][m] fp16 (raw 16-bit values): K~ row j scaled by 2^-e_j
 *   kc_mul  [B][H][cap]    fp32: 2^e_j, e_j chosen so that the row's max |value|
 *                          lands in [2^13, 2^14) (every row at full fp16 precision)
 *   v       [B][H][cap][d_v] bf16: the value cache, rows in the same order
 *
 * spa_kcache_append -- projects T new keys k [B][H][T][d] (bf16) with P
 *   [H][d][m] and writes cache rows pos .. pos+T-1 of every (b, h) (fp32
 *   products and sums, then the row exponent and fp16 rounding).  Rows are
 *   independent: appending in pieces gives the same bits as one append.
 *   SPA_ERR_SHAPE if pos + T > cap.  Asynchronous on `stream`.
 *
 * spa_attention_decode -- out[b][h][:] (fp32 [B][H][d_v]) =
 *   softmax(q~ K~^T / sqrt(m)) V over cache rows 0 .. L-1 (1 <= L <= cap), with
 *   q [B][H][d] bf16 and q~ = q P_h in fp32.  Scores, probabilities and P V are
 *   fp32.  The keys are split into chunks processed in parallel and merged by a
 *   log-sum-exp combine; the chunk results (B*H*chunks*(2+d_v) floats) and
 *   q~ (B*H*m floats) are taken on `stream` from the memory pool the library
 *   keeps per device (the one spa_attention_fwd_host uses, which keeps its
 *   reservation across synchronisations; spa_host_pool_trim releases it) and
 *   given back to it before return.  Equivalent to the last row of the causal
 *   forward over the same L keys.
 */
SPA_API int spa_kcache_append(const void *k, const void *P, void *kc, float *kc_mul, int B, int H,
                              int T, int d, int m, int pos, int cap, int dtype, void *stream);
SPA_API int spa_attention_decode(const void *q, const void *P, const void *kc, const float *kc_mul,
                                 const void *v, float *out, int B, int H, int L, int d, int m,
                                 int d_v, int cap, int dtype, void *stream);

/*
 * Sparse Feature Attention ("Scaling Attention via Feature Sparsity" notes,
 * Sec. 1 and Sec. 3): every query and key row keeps its k features of largest
 * magnitude and zeroes the rest, and attention runs on the sparsified rows,
 * softmax(Topk(Q) Topk(K)^T / sqrt(d)) V.  The dense tensor-core forward does
 * the attention (the pages' sparse-intersection kernel is a different design
 * and is not built).
 *
 * spa_topk_features -- y[r] = Topk_k(x[r]) for rows r of x [rows][d] (bf16 or
 *   fp32; y the same type; d in {32, 64, 128, 256}; 1 <= k <= d).  Ties at the
 *   k-th magnitude keep the lowest feature indices.  The selection compares
 *   the exact input values, so it is bit-exact; inputs must be finite.
 *
 * spa_sfa_attention_fwd -- out [B][H][N][d_v] fp32 = the forward above with
 *   q, k sparsified to topk features per row, i.e. spa_attention_fwd of
 *   (Topk(q), Topk(k), v) with P_h = I_d (m = d, scale 1/sqrt(d)).  d in
 *   {32, 64, 128}.  The sparsified copies, the identity P and the workspace
 *   are taken on `stream` from the library's pool and given back to it.
 */
SPA_API int spa_topk_features(const void *x, void *y, long long rows, int d, int k, int dtype,
                              void *stream);
SPA_API int spa_sfa_attention_fwd(const void *q, const void *k, const void *v, float *out, int B,
                                  int H, int N, int d, int d_v, int topk, int causal, int dtype,
                                  void *stream);

/*
 * spa_selftest_wait_timeout -- failure-detection self-test (the pages have no
 * counterpart).  Runs one small bf16 forward (B=1 H=1 N=256 d=64 m=32 d_v=64,
 * zero inputs, buffers taken and released with cudaMalloc/cudaFree on the
 * current device, default stream) in which the attention kernel withholds one
 * "scores ready" barrier arrival and limits every wait to limit_ms
 * milliseconds (1..2000).  The waiting warps give up, every role of the
 * kernel takes its abort path (drains its own copies and MMAs, frees tensor
 * memory) and the kernel sets the device error word; nothing faults or hangs.
 * The call synchronises the device, reads and clears the error word, and
 * returns SPA_ERR_TIMEOUT when the timeout was reported (the expected
 * outcome), SPA_OK when it was not, or another status if a call failed.  The
 * device stays usable afterwards.
 */
SPA_API int spa_selftest_wait_timeout(int limit_ms);

/*
 * spa_selftest_bwd_wait_timeout -- the same self-test for the fused backward
 * kernel: one small causal backward (B=1 H=1 N=256 d=64 m=32 d_v=64, zero
 * inputs) whose first "scores ready" arrival is withheld and whose waits are
 * limited to limit_ms (1..2000).  Returns SPA_ERR_TIMEOUT when the kernel
 * reported the timeout (the expected outcome), SPA_OK when it did not, or
 * another status if a call failed.  The device stays usable afterwards.
 */
SPA_API int spa_selftest_bwd_wait_timeout(int limit_ms);

/*
 * spa_selftest_proj_wait_timeout -- the same self-test for the tensor-core
 * projection kernels: the projection stage of a bf16 forward (B=1 H=8 N=4096
 * d=64, zero inputs in buffers taken and released with cudaMalloc/cudaFree;
 * m = 32 runs the per-CTA kernel, m = 64 the warp-specialised one) in which
 * CTA 0 withholds its first "product done" arrival and every wait is limited
 * to limit_ms (1..2000).  The waiting
 * threads give up, the CTA drains its copies and products, frees tensor
 * memory and sets the device error word; the other CTAs finish normally.
 * Returns SPA_ERR_TIMEOUT when the kernel reported the timeout (the expected
 * outcome), SPA_OK when it did not, SPA_ERR_SHAPE for limit_ms out of range,
 * SPA_ERR_UNSUPPORTED for another m, or another status if a call failed.
 * The device stays usable afterwards.
 */
SPA_API int spa_selftest_proj_wait_timeout(int limit_ms, int m);

/*
 * spa_selftest_copy_wait_timeout -- the same self-test for the kernels that
 * wait on their own TMA copies: kernel 0 the fused backward's row statistics
 * kernel, 1 its tensor-core finish (dq, dk, dP), 2 the SFA Top-k kernel, each
 * on zero inputs of 8 heads of 4096 rows (d = 64, m = 32, d_v = 128; Top-k on
 * 128 bf16 features, k = 16) in buffers taken and released with
 * cudaMalloc/cudaFree.  In kernels 0 and 2 CTA 0 arms its first copy
 * barrier without starting the copies; in kernel 1 CTA 0 withholds its first
 * "products done" arrival.  Every wait is limited to limit_ms (1..2000); the
 * CTA gives up, drains what it started and sets the device error word, and
 * the other CTAs finish normally.  Returns SPA_ERR_TIMEOUT when the kernel
 * reported the timeout (the expected outcome), SPA_OK when it did not,
 * SPA_ERR_SHAPE for limit_ms out of range, SPA_ERR_UNSUPPORTED for another
 * kernel number, or another status if a call failed.  The device stays usable
 * afterwards.
 */
SPA_API int spa_selftest_copy_wait_timeout(int limit_ms, int kernel);

/*
 * spa_device_error -- reads and clears the device error word of the current
 * device (synchronising it first).  *code receives 0 when no kernel gave up
 * on a bounded wait since the last call, else SPA_ERR_TIMEOUT.
 */
SPA_API int spa_device_error(int *code);

#ifdef __cplusplus
}
#endif

#endif /* SPA_H */
