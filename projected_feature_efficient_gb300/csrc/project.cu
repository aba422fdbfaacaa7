// project.cu -- the projection step  Xp = X P_h  ("Sparse Projection Attention",
// Sec. 3.1.2 and Algorithm 1 steps 2-3; "Projection-Decomposition Attention",
// Algorithm 2.1 step 1).
//
// One CTA of 128 threads owns a tile of 128 rows of one (batch, head); thread r
// computes row r.  P_h is staged in shared memory as fp32 (bf16 -> fp32 is
// exact) and read as a broadcast; X is staged 32 columns at a time.  Every
// product of two inputs is exact in fp32 and the sum is an fp32 FMA chain.
//
// Output modes:
//   F32     plain fp32 rows, [BH][N][m]  (spa_project, and the fp32 path).
//   F16X1   score-GEMM operand tiles in fp16.  To keep any input range inside
//           fp16, every Q row is divided by a power of two chosen from its own
//           max |value| (multiplier kept per row) and every 128-row K tile by a
//           power of two chosen from the tile max (multiplier kept per tile).
//           The attention kernel multiplies the raw scores back by both, which
//           is exact.  Q also carries the factor log2(e)/sqrt(m) so the scores
//           come out in base-2 logit units.
//   BF16X3  score-GEMM operand tiles in bf16, each value split v = hi + lo
//           (hi = bf16(v), lo = bf16(v - hi)); Q rows are stored [hi|hi|lo] and
//           K rows [hi|lo|hi], so one GEMM of depth 3m sums
//           hi*hi + hi*lo + lo*hi.  Used where fp16 operands are not precise
//           enough (m = 16).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.cuh"

namespace spa {
namespace {

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }

__device__ __forceinline__ float pow2i(int e) {  // e in [-126, 127]
  return __int_as_float((e + 127) << 23);
}

__device__ __forceinline__ uint16_t f16_bits(float v) { return __half_as_ushort(__float2half_rn(v)); }
__device__ __forceinline__ uint16_t bf16_bits(float v) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

// Power-of-two exponent e such that amax * 2^-e lies in [2^13, 2^14).
__device__ __forceinline__ int range_exponent(float amax) {
  if (!(amax > 0.f) || !isfinite(amax)) return 0;
  int E;
  frexpf(amax, &E);
  int e = E - 14;
  return max(-125, min(125, e));
}

template <typename T, int MP, ProjOut MODE>
__global__ void __launch_bounds__(128) project_kernel(const ProjParams p) {
  extern __shared__ float psm[];
  __shared__ float red[4];
  const int tile = blockIdx.x, bh = blockIdx.y, which = blockIdx.z;
  const int tid = threadIdx.x;
  const int d = p.d, m = p.m;
  float* Ps = psm;              // [d][MP]
  float* xs = psm + d * MP;     // [128][33]

  const T* P = static_cast<const T*>(p.P) + static_cast<size_t>(bh % p.H) * d * m;
  for (int i = tid; i < d * MP; i += 128) {
    const int l = i / MP, k = i % MP;
    Ps[i] = k < m ? to_f(P[l * m + k]) : 0.f;
  }
  const T* x = static_cast<const T*>(which == 0 ? p.x[0] : p.x[1]) + static_cast<size_t>(bh) * p.N * d;
  const int row0 = tile * kTileRows;

  float acc[MP];
#pragma unroll
  for (int k = 0; k < MP; ++k) acc[k] = 0.f;

  for (int l0 = 0; l0 < d; l0 += 32) {
    __syncthreads();
    for (int i = tid; i < kTileRows * 32; i += 128) {
      const int r = i >> 5, c = i & 31;
      const int row = row0 + r, col = l0 + c;
      xs[r * 33 + c] = (row < p.N && col < d) ? to_f(x[static_cast<size_t>(row) * d + col]) : 0.f;
    }
    __syncthreads();
    const int lmax = min(32, d - l0);
    for (int c = 0; c < lmax; ++c) {
      const float xv = xs[tid * 33 + c];
      const float* pr = Ps + (l0 + c) * MP;
#pragma unroll
      for (int k = 0; k < MP; ++k) acc[k] = fmaf(xv, pr[k], acc[k]);
    }
  }

  const int row = row0 + tid;
  if constexpr (MODE == ProjOut::F32) {
    if (row < p.N) {
      float* o = static_cast<float*>(which == 0 ? p.out[0] : p.out[1]) + (static_cast<size_t>(bh) * p.N + row) * m;
#pragma unroll
      for (int k = 0; k < MP; ++k)
        if (k < m) o[k] = acc[k];
    }
  } else {
    constexpr int KD = MODE == ProjOut::BF16X3 ? 3 * MP : MP;
    uint16_t* tout = static_cast<uint16_t*>(which == 0 ? p.out[0] : p.out[1]) +
                     (static_cast<size_t>(bh) * p.NT + tile) * (kTileRows * KD);
    const float sc = which == 0 ? p.qscale : 1.f;
#pragma unroll
    for (int k = 0; k < MP; ++k) acc[k] *= sc;

    uint16_t vals[KD];
    if constexpr (MODE == ProjOut::F16X1) {
      float amax = 0.f;
#pragma unroll
      for (int k = 0; k < MP; ++k) amax = fmaxf(amax, fabsf(acc[k]));
      if (which == 1) {  // one exponent for the whole K tile
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if ((tid & 31) == 0) red[tid >> 5] = amax;
        __syncthreads();
        amax = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
      }
      const int e = range_exponent(amax);
      const float down = pow2i(-e);
#pragma unroll
      for (int k = 0; k < MP; ++k) vals[k] = f16_bits(acc[k] * down);
      if (which == 0)
        p.mul[0][static_cast<size_t>(bh) * p.NT * kTileRows + row] = pow2i(e);
      else if (tid == 0)
        p.mul[1][static_cast<size_t>(bh) * p.NT + tile] = pow2i(e);
    } else {
#pragma unroll
      for (int k = 0; k < MP; ++k) {
        const __nv_bfloat16 hi = __float2bfloat16_rn(acc[k]);
        const uint16_t hib = __bfloat16_as_ushort(hi);
        const uint16_t lob = bf16_bits(acc[k] - __bfloat162float(hi));
        vals[k] = hib;                                   // segment 0: hi for both
        vals[MP + k] = which == 0 ? hib : lob;           // Q: hi, K: lo
        vals[2 * MP + k] = which == 0 ? lob : hib;       // Q: lo, K: hi
      }
      if (which == 0)
        p.mul[0][static_cast<size_t>(bh) * p.NT * kTileRows + row] = 1.f;
      else if (tid == 0)
        p.mul[1][static_cast<size_t>(bh) * p.NT + tile] = 1.f;
    }
    // interleaved core-matrix layout: 8 columns (16 bytes) per store
#pragma unroll
    for (int c8 = 0; c8 < KD / 8; ++c8) {
      uint4 w;
      w.x = vals[c8 * 8 + 0] | (static_cast<uint32_t>(vals[c8 * 8 + 1]) << 16);
      w.y = vals[c8 * 8 + 2] | (static_cast<uint32_t>(vals[c8 * 8 + 3]) << 16);
      w.z = vals[c8 * 8 + 4] | (static_cast<uint32_t>(vals[c8 * 8 + 5]) << 16);
      w.w = vals[c8 * 8 + 6] | (static_cast<uint32_t>(vals[c8 * 8 + 7]) << 16);
      *reinterpret_cast<uint4*>(tout + (c8 * 16 + (tid >> 3)) * 64 + (tid & 7) * 8) = w;
    }
  }
}

template <typename T, int MP, ProjOut MODE>
cudaError_t launch_one(const ProjParams& p, cudaStream_t stream) {
  const size_t smem = (static_cast<size_t>(p.d) * MP + kTileRows * 33) * sizeof(float);
  auto kern = project_kernel<T, MP, MODE>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  dim3 grid(p.NT, p.BH, p.nx);
  kern<<<grid, 128, smem, stream>>>(p);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_f32_out(const ProjParams& p, cudaStream_t stream) {
  if (p.m <= 16) return launch_one<T, 16, ProjOut::F32>(p, stream);
  if (p.m <= 32) return launch_one<T, 32, ProjOut::F32>(p, stream);
  if (p.m <= 64) return launch_one<T, 64, ProjOut::F32>(p, stream);
  return launch_one<T, 128, ProjOut::F32>(p, stream);
}

}  // namespace

cudaError_t launch_project(const ProjParams& p, cudaStream_t stream) {
  if (p.mode == ProjOut::F32)
    return p.bf16_in ? launch_f32_out<__nv_bfloat16>(p, stream) : launch_f32_out<float>(p, stream);
  if (!p.bf16_in) return cudaErrorInvalidValue;
  if (p.mode == ProjOut::BF16X3) {
    if (p.m == 16) return launch_one<__nv_bfloat16, 16, ProjOut::BF16X3>(p, stream);
    return cudaErrorInvalidValue;
  }
  switch (p.m) {
    case 32: return launch_one<__nv_bfloat16, 32, ProjOut::F16X1>(p, stream);
    case 64: return launch_one<__nv_bfloat16, 64, ProjOut::F16X1>(p, stream);
    case 128: return launch_one<__nv_bfloat16, 128, ProjOut::F16X1>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace spa
