// bwd_simt.cu -- the backward of projected-feature attention on CUDA cores,
// for the shapes the tensor-core kernels do not cover (fp32 inputs, which the
// fp32 tolerance needs in true fp32; bf16 with m = 128, whose accumulators do
// not fit the fused kernel's tensor memory).
//
// The gradients follow the chain rule of the forward ("Sparse Projection
// Attention", Sec. 3.4.1: the gradient reaches Q through Qp and the projection
// through Q^T dQp), with the logits s_ij = <Qp_i, Kp_j> / sqrt(m), the
// forward's row log-sum-exp L_i and D_i = <dO_i, O_i>:
//   A_ij = exp(s_ij - L_i)                (recomputed, never stored)
//   dV_j  = sum_i A_ij dO_i
//   dS_ij = A_ij (<dO_i, V_j> - D_i) / sqrt(m)
//   dKp_j = sum_i dS_ij Qp_i,   dQp_i = sum_j dS_ij Kp_j
//   dq = dQp P_h^T,  dk = dKp P_h^T,  dP_h = sum_b (q^T dQp + k^T dKp)
// Flash-style: no N x N block is written; every product is recomputed where
// it is needed, in fp32.  One warp walks one key row (dV, dKp) or one query
// row (dQp), its lanes splitting the feature columns; the projection gradient
// dP_h is reduced over fixed row chunks and then over the chunks in order, so
// the result does not depend on scheduling.
#include <cuda_bf16.h>

#include "kernels.cuh"

namespace spa {
namespace {

constexpr int kWarps = 4;  // warps per block of the row kernels
constexpr int kMaxM = 128, kMaxDv = 256;

template <typename T>
__device__ __forceinline__ float ld(const T* p, size_t i);
template <>
__device__ __forceinline__ float ld<float>(const float* p, size_t i) {
  return __ldg(p + i);
}
template <>
__device__ __forceinline__ float ld<__nv_bfloat16>(const __nv_bfloat16* p, size_t i) {
  return __bfloat162float(p[i]);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// D_i = <dO_i, O_i>: one warp per row
template <typename T>
__global__ void simt_dsum_kernel(const T* __restrict__ dO, const float* __restrict__ out,
                                 float* __restrict__ dsum, long long rows, int dv) {
  const long long row = static_cast<long long>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float acc = 0.f;
  for (int c = lane; c < dv; c += 32)
    acc = fmaf(ld(dO, static_cast<size_t>(row) * dv + c), out[static_cast<size_t>(row) * dv + c], acc);
  acc = warp_sum(acc);
  if (lane == 0) dsum[row] = acc;
}

// dV_j and dKp_j: one warp per key row j of one (batch, head)
template <typename T>
__global__ void simt_dkv_kernel(BwdSimtParams p) {
  constexpr int CM = kMaxM / 32, CV = kMaxDv / 32;  // columns per lane at most
  const int bh = blockIdx.y;
  const int j = blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (j >= p.N) return;
  const T* dO = static_cast<const T*>(p.dO);
  const T* v = static_cast<const T*>(p.v);
  const size_t base = static_cast<size_t>(bh) * p.N;
  const float scale = rsqrtf(static_cast<float>(p.m));
  float kj[CM], vj[CV], dvj[CV], dkj[CM];
#pragma unroll
  for (int t = 0; t < CM; ++t) {
    const int c = lane + 32 * t;
    kj[t] = c < p.m ? p.kp[(base + j) * p.m + c] : 0.f;
    dkj[t] = 0.f;
  }
#pragma unroll
  for (int t = 0; t < CV; ++t) {
    const int c = lane + 32 * t;
    vj[t] = c < p.dv ? ld(v, (base + j) * p.dv + c) : 0.f;
    dvj[t] = 0.f;
  }
  for (int i = p.causal ? j : 0; i < p.N; ++i) {
    float s = 0.f, dp = 0.f, qi[CM], gi[CV];
#pragma unroll
    for (int t = 0; t < CM; ++t) {
      const int c = lane + 32 * t;
      qi[t] = c < p.m ? p.qp[(base + i) * p.m + c] : 0.f;
      s = fmaf(qi[t], kj[t], s);
    }
#pragma unroll
    for (int t = 0; t < CV; ++t) {
      const int c = lane + 32 * t;
      gi[t] = c < p.dv ? ld(dO, (base + i) * p.dv + c) : 0.f;
      dp = fmaf(gi[t], vj[t], dp);
    }
    s = warp_sum(s);
    dp = warp_sum(dp);
    const float a = expf(s * scale - p.lse[base + i]);
    const float ds = a * (dp - p.dsum[base + i]) * scale;
#pragma unroll
    for (int t = 0; t < CV; ++t) dvj[t] = fmaf(a, gi[t], dvj[t]);
#pragma unroll
    for (int t = 0; t < CM; ++t) dkj[t] = fmaf(ds, qi[t], dkj[t]);
  }
#pragma unroll
  for (int t = 0; t < CV; ++t) {
    const int c = lane + 32 * t;
    if (c < p.dv) p.dv_out[(base + j) * p.dv + c] = dvj[t];
  }
#pragma unroll
  for (int t = 0; t < CM; ++t) {
    const int c = lane + 32 * t;
    if (c < p.m) p.dkp[(base + j) * p.m + c] = dkj[t];
  }
}

// dQp_i: one warp per query row i of one (batch, head)
template <typename T>
__global__ void simt_dq_kernel(BwdSimtParams p) {
  constexpr int CM = kMaxM / 32, CV = kMaxDv / 32;
  const int bh = blockIdx.y;
  const int i = blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (i >= p.N) return;
  const T* dO = static_cast<const T*>(p.dO);
  const T* v = static_cast<const T*>(p.v);
  const size_t base = static_cast<size_t>(bh) * p.N;
  const float scale = rsqrtf(static_cast<float>(p.m));
  const float Li = p.lse[base + i], Di = p.dsum[base + i];
  float qi[CM], gi[CV], dqi[CM];
#pragma unroll
  for (int t = 0; t < CM; ++t) {
    const int c = lane + 32 * t;
    qi[t] = c < p.m ? p.qp[(base + i) * p.m + c] : 0.f;
    dqi[t] = 0.f;
  }
#pragma unroll
  for (int t = 0; t < CV; ++t) {
    const int c = lane + 32 * t;
    gi[t] = c < p.dv ? ld(dO, (base + i) * p.dv + c) : 0.f;
  }
  const int jend = p.causal ? i + 1 : p.N;
  for (int j = 0; j < jend; ++j) {
    float s = 0.f, dp = 0.f, kj[CM];
#pragma unroll
    for (int t = 0; t < CM; ++t) {
      const int c = lane + 32 * t;
      kj[t] = c < p.m ? p.kp[(base + j) * p.m + c] : 0.f;
      s = fmaf(qi[t], kj[t], s);
    }
#pragma unroll
    for (int t = 0; t < CV; ++t) {
      const int c = lane + 32 * t;
      if (c < p.dv) dp = fmaf(gi[t], ld(v, (base + j) * p.dv + c), dp);
    }
    s = warp_sum(s);
    dp = warp_sum(dp);
    const float ds = expf(s * scale - Li) * (dp - Di) * scale;
#pragma unroll
    for (int t = 0; t < CM; ++t) dqi[t] = fmaf(ds, kj[t], dqi[t]);
  }
#pragma unroll
  for (int t = 0; t < CM; ++t) {
    const int c = lane + 32 * t;
    if (c < p.m) p.dqp[(base + i) * p.m + c] = dqi[t];
  }
}

// dx[bh][i][l] = sum_c g[bh][i][c] P[h][l][c]: one thread per (row, l)
template <typename T>
__global__ void simt_back_project_kernel(const float* __restrict__ g, const T* __restrict__ P,
                                         float* __restrict__ dx, long long rows, int H, int N,
                                         int d, int m) {
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= rows * d) return;
  const long long row = t / d;
  const int l = static_cast<int>(t % d);
  const int h = static_cast<int>((row / N) % H);
  const float* gr = g + row * m;
  const size_t pr = (static_cast<size_t>(h) * d + l) * m;
  float acc = 0.f;
  for (int c = 0; c < m; ++c) acc = fmaf(gr[c], ld(P, pr + c), acc);
  dx[t] = acc;
}

// part[h][chunk][l][c] = sum over the chunk's rows (b, i) of
// q[b,h,i,l] dQp[b,h,i,c] + k[b,h,i,l] dKp[b,h,i,c]
template <typename T>
__global__ void simt_dp_partial_kernel(BwdSimtParams p, int rows_per_chunk) {
  const int h = blockIdx.y, chunk = blockIdx.z;
  const T* q = static_cast<const T*>(p.q);
  const T* k = static_cast<const T*>(p.k);
  const long long rows = static_cast<long long>(p.B) * p.N;
  const long long r0 = static_cast<long long>(chunk) * rows_per_chunk;
  const long long r1 = r0 + rows_per_chunk < rows ? r0 + rows_per_chunk : rows;
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < p.d * p.m; e += gridDim.x * blockDim.x) {
    const int l = e / p.m, c = e % p.m;
    float acc = 0.f;
    for (long long r = r0; r < r1; ++r) {
      const long long b = r / p.N, i = r % p.N;
      const size_t row = (static_cast<size_t>(b) * p.H + h) * p.N + i;
      acc = fmaf(ld(q, row * p.d + l), p.dqp[row * p.m + c], acc);
      acc = fmaf(ld(k, row * p.d + l), p.dkp[row * p.m + c], acc);
    }
    p.part[(static_cast<size_t>(h) * p.chunks + chunk) * p.d * p.m + e] = acc;
  }
}

__global__ void simt_dp_reduce_kernel(const float* __restrict__ part, float* __restrict__ dP,
                                      int H, int chunks, int dm) {
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= static_cast<long long>(H) * dm) return;
  const int h = static_cast<int>(t / dm), e = static_cast<int>(t % dm);
  float acc = 0.f;
  for (int c = 0; c < chunks; ++c) acc += part[(static_cast<size_t>(h) * chunks + c) * dm + e];
  dP[t] = acc;
}

unsigned blocks_for(long long n, int per) { return static_cast<unsigned>((n + per - 1) / per); }

template <typename T>
cudaError_t launch_typed(const BwdSimtParams& p, cudaStream_t s) {
  const int BH = p.B * p.H;
  const long long rows = static_cast<long long>(BH) * p.N;
  simt_dsum_kernel<T><<<blocks_for(rows, kWarps), 32 * kWarps, 0, s>>>(
      static_cast<const T*>(p.dO), p.out, p.dsum, rows, p.dv);
  const dim3 grid(blocks_for(p.N, kWarps), BH);
  simt_dkv_kernel<T><<<grid, 32 * kWarps, 0, s>>>(p);
  simt_dq_kernel<T><<<grid, 32 * kWarps, 0, s>>>(p);
  simt_back_project_kernel<T><<<blocks_for(rows * p.d, 256), 256, 0, s>>>(
      p.dqp, static_cast<const T*>(p.P), p.dq, rows, p.H, p.N, p.d, p.m);
  simt_back_project_kernel<T><<<blocks_for(rows * p.d, 256), 256, 0, s>>>(
      p.dkp, static_cast<const T*>(p.P), p.dk, rows, p.H, p.N, p.d, p.m);
  const long long per_chunk = (static_cast<long long>(p.B) * p.N + p.chunks - 1) / p.chunks;
  const dim3 pgrid(blocks_for(static_cast<long long>(p.d) * p.m, 256), p.H, p.chunks);
  simt_dp_partial_kernel<T><<<pgrid, 256, 0, s>>>(p, static_cast<int>(per_chunk));
  simt_dp_reduce_kernel<<<blocks_for(static_cast<long long>(p.H) * p.d * p.m, 256), 256, 0, s>>>(
      p.part, p.dP, p.H, p.chunks, p.d * p.m);
  return cudaGetLastError();
}

}  // namespace

int bwd_simt_chunks(int B, int N) {
  const long long rows = static_cast<long long>(B) * N;
  const long long c = (rows + 1023) / 1024;
  return static_cast<int>(c < 1 ? 1 : (c > 256 ? 256 : c));
}

cudaError_t launch_bwd_simt(const BwdSimtParams& p, cudaStream_t stream) {
  if (p.m < 1 || p.m > kMaxM || p.dv < 1 || p.dv > kMaxDv || p.chunks < 1)
    return cudaErrorInvalidValue;
  if (static_cast<long long>(p.B) * p.H * p.N == 0) return cudaSuccess;
  return p.bf16 ? launch_typed<__nv_bfloat16>(p, stream) : launch_typed<float>(p, stream);
}

}  // namespace spa
