// backward.cu -- gradients of the projected-feature attention forward
// ("Sparse Projection Attention", Sec. 3.4.1 and Algorithm 2: the projection
// is trained through these gradients).  Per (batch b, head h), with the
// forward's softmax A = softmax(Qp Kp^T / sqrt(m)) (causal mask j <= i):
//   dV  = A^T dO
//   dA  = dO V^T,   D_i = <dO_i, O_i>,   dS = A * (dA - D) / sqrt(m)
//   dQp = dS Kp,    dKp = dS^T Qp
//   dQ  = dQp P_h^T,  dK = dKp P_h^T,  dP_h = sum_b (Q^T dQp + K^T dKp)
//
// This file holds the general version (fp32 inputs, and shapes the fused
// tensor-core backward in bwd_ws.cu does not cover).  It materialises A and dS
// for a group of heads at a time: the
// products are plain library GEMMs (cuBLAS, fp32 accumulation; TF32 products
// for bf16 inputs, whose values TF32 holds exactly; full fp32 for fp32
// inputs) and the element-wise steps (conversion, the row dot D, the masked
// softmax, dS, the batch sum of dP) are the kernels below.  It is HBM-bound on
// the N x N blocks.  The file also holds the library products that turn the
// fused backward's dQp / dKp into dq, dk and dP (run_backward_post).
#include <cublas_v2.h>
#include <cuda_bf16.h>
#include <math.h>

#include <mutex>

#include "kernels.cuh"

namespace spa {
namespace {

__global__ void to_f32_kernel(const void* src, float* dst, long long n, int bf16) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  dst[i] = bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(src)[i])
                : static_cast<const float*>(src)[i];
}

// D[r] = <dO[r], O[r]>: one warp per row
__global__ void rowdot_kernel(const float* dO, const float* O, float* D, long long rows, int dv) {
  const long long r = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (r >= rows) return;
  const int lane = threadIdx.x & 31;
  float acc = 0.f;
  for (int c = lane; c < dv; c += 32) acc = fmaf(dO[r * dv + c], O[r * dv + c], acc);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) D[r] = acc;
}

__device__ __forceinline__ float block_reduce(float v, float* sh, bool is_max) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float w = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? fmaxf(v, w) : v + w;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  float r = sh[0];
  for (int w = 1; w < static_cast<int>(blockDim.x >> 5); ++w) r = is_max ? fmaxf(r, sh[w]) : r + sh[w];
  return r;
}

// S row r (query i = r % N of its head) -> A = softmax(S * scale) over keys
// j <= i (causal) or all j; masked entries become 0.  One CTA per row.
__global__ void softmax_rows_kernel(float* S, int N, float scale, int causal) {
  __shared__ float sh[32];
  const long long r = blockIdx.x;
  const int i = static_cast<int>(r % N);
  const int nk = causal ? i + 1 : N;
  float* row = S + r * N;
  float mx = -INFINITY;
  for (int j = threadIdx.x; j < nk; j += blockDim.x) mx = fmaxf(mx, row[j] * scale);
  mx = block_reduce(mx, sh, true);
  float sum = 0.f;
  for (int j = threadIdx.x; j < nk; j += blockDim.x) {
    const float e = expf(row[j] * scale - mx);
    row[j] = e;
    sum += e;
  }
  sum = block_reduce(sum, sh, false);
  const float inv = 1.f / sum;
  for (int j = threadIdx.x; j < N; j += blockDim.x) row[j] = j < nk ? row[j] * inv : 0.f;
}

// dA row r -> dS = A * (dA - D_i) * scale (A is 0 where masked)
__global__ void ds_rows_kernel(const float* A, float* dA, const float* D, int N, float scale) {
  const long long r = blockIdx.x;
  const float d = D[r];
  const float* a = A + r * N;
  float* g = dA + r * N;
  for (int j = threadIdx.x; j < N; j += blockDim.x) g[j] = a[j] * (g[j] - d) * scale;
}

// Row-major C[M x N] = alpha op(A)[M x K] op(B)[K x N] + beta C, batched with
// element strides; lda/ldb/ldc are the row lengths of A, B, C as stored.
// (cuBLAS is column-major: it computes C^T = op(B)^T op(A)^T.)
cublasStatus_t gemm_rm(cublasHandle_t h, bool ta, bool tb, int M, int N, int K, const float* A,
                       int lda, long long sA, const float* B, int ldb, long long sB, float* C,
                       int ldc, long long sC, int batch, float alpha, float beta,
                       cublasComputeType_t ct) {
  return cublasGemmStridedBatchedEx(h, tb ? CUBLAS_OP_T : CUBLAS_OP_N, ta ? CUBLAS_OP_T : CUBLAS_OP_N,
                                    N, M, K, &alpha, B, CUDA_R_32F, ldb, sB, A, CUDA_R_32F, lda, sA,
                                    &beta, C, CUDA_R_32F, ldc, sC, batch, ct, CUBLAS_GEMM_DEFAULT);
}

// The same with bf16 A and B (fp32 accumulation and output).
cublasStatus_t gemm_rm_bf16(cublasHandle_t h, bool ta, bool tb, int M, int N, int K, const void* A,
                            int lda, long long sA, const void* B, int ldb, long long sB, float* C,
                            int ldc, long long sC, int batch, float alpha, float beta) {
  return cublasGemmStridedBatchedEx(h, tb ? CUBLAS_OP_T : CUBLAS_OP_N, ta ? CUBLAS_OP_T : CUBLAS_OP_N,
                                    N, M, K, &alpha, B, CUDA_R_16BF, ldb, sB, A, CUDA_R_16BF, lda, sA,
                                    &beta, C, CUDA_R_32F, ldc, sC, batch, CUBLAS_COMPUTE_32F,
                                    CUBLAS_GEMM_DEFAULT);
}

std::mutex g_blas_mutex;
cublasHandle_t g_blas[64] = {};

// The device's handle, bound to `stream`; the caller holds g_blas_mutex.
cublasHandle_t blas_handle(cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!g_blas[dev] && cublasCreate(&g_blas[dev]) != CUBLAS_STATUS_SUCCESS) return nullptr;
  if (cublasSetStream(g_blas[dev], stream) != CUBLAS_STATUS_SUCCESS) return nullptr;
  return g_blas[dev];
}

}  // namespace

size_t backward_workspace_bytes(const BwdParams& p) {
  const size_t BH = static_cast<size_t>(p.B) * p.H, N = p.N;
  const size_t f = sizeof(float);
  auto al = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  size_t t = 0;
  t += 2 * al(BH * N * p.d * f);        // q, k as fp32
  t += 2 * al(BH * N * p.dv * f);       // v, dO as fp32
  t += al(static_cast<size_t>(p.H) * p.d * p.m * f);  // P as fp32
  t += 4 * al(BH * N * p.m * f);        // Qp, Kp, dQp, dKp
  t += al(BH * N * f);                  // D
  t += 2 * al(static_cast<size_t>(p.group) * N * N * f);  // A and dA / dS of a head group
  return t;
}

int backward_group(int B, int H, int N, size_t budget_bytes) {
  const size_t per = 2ull * N * N * sizeof(float);
  long long g = per ? static_cast<long long>(budget_bytes / per) : 1;
  if (g < 1) g = 1;
  if (g > static_cast<long long>(B) * H) g = static_cast<long long>(B) * H;
  return static_cast<int>(g);
}

// Returns 0, or -1 for a CUDA error, -2 for a cuBLAS error.
int run_backward(const BwdParams& p, void* ws, cudaStream_t stream) {
  std::lock_guard<std::mutex> lock(g_blas_mutex);  // one handle per device, one user at a time
  cublasHandle_t h = blas_handle(stream);
  if (!h) return -2;
  const cublasComputeType_t ct = p.bf16 ? CUBLAS_COMPUTE_32F_FAST_TF32 : CUBLAS_COMPUTE_32F;

  const long long BH = static_cast<long long>(p.B) * p.H, N = p.N;
  const int d = p.d, m = p.m, dv = p.dv;
  auto al = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  char* w = static_cast<char*>(ws);
  auto take = [&](size_t bytes) {
    float* r = reinterpret_cast<float*>(w);
    w += al(bytes);
    return r;
  };
  float* q32 = take(BH * N * d * 4);
  float* k32 = take(BH * N * d * 4);
  float* v32 = take(BH * N * dv * 4);
  float* dO32 = take(BH * N * dv * 4);
  float* P32 = take(static_cast<size_t>(p.H) * d * m * 4);
  float* qp = take(BH * N * m * 4);
  float* kp = take(BH * N * m * 4);
  float* dqp = take(BH * N * m * 4);
  float* dkp = take(BH * N * m * 4);
  float* D = take(BH * N * 4);
  float* Abuf = take(static_cast<size_t>(p.group) * N * N * 4);
  float* Gbuf = take(static_cast<size_t>(p.group) * N * N * 4);

  auto conv = [&](const void* src, float* dst, long long n) {
    if (n == 0) return true;
    to_f32_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(src, dst, n, p.bf16);
    return cudaGetLastError() == cudaSuccess;
  };
  if (!conv(p.q, q32, BH * N * d) || !conv(p.k, k32, BH * N * d) || !conv(p.v, v32, BH * N * dv) ||
      !conv(p.dO, dO32, BH * N * dv) || !conv(p.P, P32, static_cast<long long>(p.H) * d * m))
    return -1;
  // D_i = <dO_i, O_i>
  rowdot_kernel<<<static_cast<unsigned>((BH * N + 7) / 8), 256, 0, stream>>>(dO32, p.out, D, BH * N, dv);
  if (cudaGetLastError() != cudaSuccess) return -1;

  // Qp = q P_h, Kp = k P_h: per batch entry, batched over heads
  for (int b = 0; b < p.B; ++b) {
    const long long o = static_cast<long long>(b) * p.H * N;
    if (gemm_rm(h, false, false, N, m, d, q32 + o * d, d, N * d, P32, m, static_cast<long long>(d) * m,
                qp + o * m, m, N * m, p.H, 1.f, 0.f, ct) != CUBLAS_STATUS_SUCCESS ||
        gemm_rm(h, false, false, N, m, d, k32 + o * d, d, N * d, P32, m, static_cast<long long>(d) * m,
                kp + o * m, m, N * m, p.H, 1.f, 0.f, ct) != CUBLAS_STATUS_SUCCESS)
      return -2;
  }
  const float rsm = static_cast<float>(1.0 / std::sqrt(static_cast<double>(m)));
  for (long long g0 = 0; g0 < BH; g0 += p.group) {
    const int G = static_cast<int>(BH - g0 < p.group ? BH - g0 : p.group);
    const long long NN = N * N;
    // A = softmax(Qp Kp^T / sqrt(m)) (masked)
    if (gemm_rm(h, false, true, N, N, m, qp + g0 * N * m, m, N * m, kp + g0 * N * m, m, N * m, Abuf,
                N, NN, G, 1.f, 0.f, ct) != CUBLAS_STATUS_SUCCESS)
      return -2;
    softmax_rows_kernel<<<static_cast<unsigned>(G * N), 256, 0, stream>>>(Abuf, N, rsm, p.causal);
    if (cudaGetLastError() != cudaSuccess) return -1;
    // dA = dO V^T, then dS = A * (dA - D) / sqrt(m)
    if (gemm_rm(h, false, true, N, N, dv, dO32 + g0 * N * dv, dv, N * dv, v32 + g0 * N * dv, dv,
                N * dv, Gbuf, N, NN, G, 1.f, 0.f, ct) != CUBLAS_STATUS_SUCCESS)
      return -2;
    ds_rows_kernel<<<static_cast<unsigned>(G * N), 256, 0, stream>>>(Abuf, Gbuf, D + g0 * N, N, rsm);
    if (cudaGetLastError() != cudaSuccess) return -1;
    // dQp = dS Kp, dKp = dS^T Qp, dV = A^T dO
    if (gemm_rm(h, false, false, N, m, N, Gbuf, N, NN, kp + g0 * N * m, m, N * m, dqp + g0 * N * m,
                m, N * m, G, 1.f, 0.f, ct) != CUBLAS_STATUS_SUCCESS ||
        gemm_rm(h, true, false, N, m, N, Gbuf, N, NN, qp + g0 * N * m, m, N * m, dkp + g0 * N * m, m,
                N * m, G, 1.f, 0.f, ct) != CUBLAS_STATUS_SUCCESS ||
        gemm_rm(h, true, false, N, dv, N, Abuf, N, NN, dO32 + g0 * N * dv, dv, N * dv,
                p.dv_out + g0 * N * dv, dv, N * dv, G, 1.f, 0.f, ct) != CUBLAS_STATUS_SUCCESS)
      return -2;
  }
  // dQ = dQp P_h^T, dK = dKp P_h^T; dP_h = sum_b q^T dQp + k^T dKp
  for (int b = 0; b < p.B; ++b) {
    const long long o = static_cast<long long>(b) * p.H * N;
    const float beta = b == 0 ? 0.f : 1.f;
    if (gemm_rm(h, false, true, N, d, m, dqp + o * m, m, N * m, P32, m, static_cast<long long>(d) * m,
                p.dq + o * d, d, N * d, p.H, 1.f, 0.f, ct) != CUBLAS_STATUS_SUCCESS ||
        gemm_rm(h, false, true, N, d, m, dkp + o * m, m, N * m, P32, m, static_cast<long long>(d) * m,
                p.dk + o * d, d, N * d, p.H, 1.f, 0.f, ct) != CUBLAS_STATUS_SUCCESS ||
        gemm_rm(h, true, false, d, m, N, q32 + o * d, d, N * d, dqp + o * m, m, N * m, p.dP, m,
                static_cast<long long>(d) * m, p.H, 1.f, beta, ct) != CUBLAS_STATUS_SUCCESS ||
        gemm_rm(h, true, false, d, m, N, k32 + o * d, d, N * d, dkp + o * m, m, N * m, p.dP, m,
                static_cast<long long>(d) * m, p.H, 1.f, 1.f, ct) != CUBLAS_STATUS_SUCCESS)
      return -2;
  }
  return 0;
}

// The projection's share of the fused backward.  xq, xk hold dQp and dKp as
// bf16 pairs [hi | lo] per row ([BH][N][2m]; hi + lo carries 16 significant
// bits), P2[h] = [P_h | P_h] ([H][d][2m]), so that
//   dq = xq P2^T = dQp P_h^T,   dk = xk P2^T = dKp P_h^T,
//   R_h = sum_b q^T xq + k^T xk  ([H][d][2m]),  dP_h = R_h[:, :m] + R_h[:, m:].
// Every product is a plain bf16 GEMM with fp32 accumulation.
int run_backward_post(const void* q, const void* k, const uint16_t* P2, const uint16_t* xq,
                      const uint16_t* xk, float* R, float* dq, float* dk, float* dP, int B,
                      int H, int N, int d, int m, cudaStream_t stream) {
  std::lock_guard<std::mutex> lock(g_blas_mutex);
  cublasHandle_t h = blas_handle(stream);
  if (!h) return -2;
  const long long Nl = N, m2 = 2 * m;
  const auto* qb = static_cast<const uint16_t*>(q);
  const auto* kb = static_cast<const uint16_t*>(k);
  for (int b = 0; b < B; ++b) {
    const long long o = static_cast<long long>(b) * H * Nl;
    if (gemm_rm_bf16(h, false, true, N, d, static_cast<int>(m2), xq + o * m2, static_cast<int>(m2),
                     Nl * m2, P2, static_cast<int>(m2), static_cast<long long>(d) * m2, dq + o * d, d,
                     Nl * d, H, 1.f, 0.f) != CUBLAS_STATUS_SUCCESS ||
        gemm_rm_bf16(h, false, true, N, d, static_cast<int>(m2), xk + o * m2, static_cast<int>(m2),
                     Nl * m2, P2, static_cast<int>(m2), static_cast<long long>(d) * m2, dk + o * d, d,
                     Nl * d, H, 1.f, 0.f) != CUBLAS_STATUS_SUCCESS ||
        gemm_rm_bf16(h, true, false, d, static_cast<int>(m2), N, qb + o * d, d, Nl * d, xq + o * m2,
                     static_cast<int>(m2), Nl * m2, R, static_cast<int>(m2),
                     static_cast<long long>(d) * m2, H, 1.f, b == 0 ? 0.f : 1.f) !=
            CUBLAS_STATUS_SUCCESS ||
        gemm_rm_bf16(h, true, false, d, static_cast<int>(m2), N, kb + o * d, d, Nl * d, xk + o * m2,
                     static_cast<int>(m2), Nl * m2, R, static_cast<int>(m2),
                     static_cast<long long>(d) * m2, H, 1.f, 1.f) != CUBLAS_STATUS_SUCCESS)
      return -2;
  }
  return launch_bwd_fold(R, dP, H, d, m, stream) == cudaSuccess ? 0 : -1;
}

}  // namespace spa
