// topk.cu -- row-wise Top-k feature sparsification (Sparse Feature Attention
// notes, Sec. 1 "feature sparsification": every query / key row keeps its k
// coordinates of largest magnitude and zeroes the rest; attention then runs
// on the sparsified rows at scale 1/sqrt(d)).
//
// One warp per row of d = 32 * E features; lane l holds the E consecutive
// features E*l .. E*l + E - 1.  The k-th largest magnitude T is found by a
// binary search over the magnitude's bit pattern (for non-negative floats the
// bit pattern orders like the value), counting with warp sums.  Every
// feature with |x| > T is kept, and of the features with |x| == T the ones
// with the lowest indices, as many as k still needs (a warp-wide exclusive
// scan in index order).  The selection is made on the exact input values, so
// it is bit-exact and deterministic.
#include <cuda_bf16.h>
#include <stdint.h>

#include "kernels.cuh"

namespace spa {
namespace {

template <typename T>
struct Mag;
template <>
struct Mag<float> {
  static __device__ __forceinline__ uint32_t bits(float v) { return __float_as_uint(v) & 0x7fffffffu; }
  static constexpr int kBits = 31;
};
template <>
struct Mag<__nv_bfloat16> {
  static __device__ __forceinline__ uint32_t bits(__nv_bfloat16 v) {
    return static_cast<uint32_t>(__bfloat16_as_ushort(v)) & 0x7fffu;
  }
  static constexpr int kBits = 15;
};

__device__ __forceinline__ int warp_sum(int v) {
  return static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(v)));
}

template <typename T, int E>
__global__ void __launch_bounds__(256) topk_rows_kernel(const T* __restrict__ x, T* __restrict__ y,
                                                        long long rows, int k) {
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  const T* xr = x + row * (32 * E) + lane * E;
  T* yr = y + row * (32 * E) + lane * E;
  T v[E];
  uint32_t mag[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    v[e] = xr[e];
    mag[e] = Mag<T>::bits(v[e]);
  }
  // largest T with count(|x| >= T) >= k: set the threshold's bits from the top
  uint32_t t = 0;
  for (int b = Mag<T>::kBits - 1; b >= 0; --b) {
    const uint32_t cand = t | (1u << b);
    int c = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) c += mag[e] >= cand ? 1 : 0;
    if (warp_sum(c) >= k) t = cand;
  }
  int above = 0, ties = 0;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    above += mag[e] > t ? 1 : 0;
    ties += mag[e] == t ? 1 : 0;
  }
  const int need = k - warp_sum(above);  // ties to keep, lowest feature index first
  int before = ties;                      // exclusive scan of ties over lanes
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, before, o);
    if (lane >= o) before += n;
  }
  before -= ties;
  const T zero = T(0.f);
#pragma unroll
  for (int e = 0; e < E; ++e) {
    bool keep = mag[e] > t;
    if (mag[e] == t) {
      keep = before < need;
      ++before;
    }
    yr[e] = keep ? v[e] : zero;
  }
}

template <typename T>
cudaError_t launch_typed(const TopkParams& p, cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>((p.rows + 7) / 8);
  const T* x = static_cast<const T*>(p.x);
  T* y = static_cast<T*>(p.y);
  switch (p.d) {
    case 32: topk_rows_kernel<T, 1><<<grid, 256, 0, stream>>>(x, y, p.rows, p.k); break;
    case 64: topk_rows_kernel<T, 2><<<grid, 256, 0, stream>>>(x, y, p.rows, p.k); break;
    case 128: topk_rows_kernel<T, 4><<<grid, 256, 0, stream>>>(x, y, p.rows, p.k); break;
    case 256: topk_rows_kernel<T, 8><<<grid, 256, 0, stream>>>(x, y, p.rows, p.k); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// P = I_d for every head, so that the forward runs on the sparsified rows
// unchanged (Q I = Q exactly) at scale 1/sqrt(d).
template <typename T>
__global__ void identity_kernel(T* P, long long n, int d) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int c = static_cast<int>(i % d), l = static_cast<int>((i / d) % d);
  P[i] = T(l == c ? 1.f : 0.f);
}

}  // namespace

cudaError_t launch_identity(void* P, int H, int d, int bf16, cudaStream_t stream) {
  const long long n = static_cast<long long>(H) * d * d;
  if (n == 0) return cudaSuccess;
  const unsigned grid = static_cast<unsigned>((n + 255) / 256);
  if (bf16)
    identity_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(static_cast<__nv_bfloat16*>(P), n, d);
  else
    identity_kernel<float><<<grid, 256, 0, stream>>>(static_cast<float*>(P), n, d);
  return cudaGetLastError();
}

cudaError_t launch_topk(const TopkParams& p, cudaStream_t stream) {
  if (p.rows == 0) return cudaSuccess;
  if (p.rows > 8LL * 0x7fffffffLL) return cudaErrorInvalidValue;
  return p.bf16 ? launch_typed<__nv_bfloat16>(p, stream) : launch_typed<float>(p, stream);
}

}  // namespace spa
