// decode.cu -- the projected key cache and single-query (decode) attention.
//
// The projection is what makes the cache small: a decode step needs only
// K~ = K P_h (m values per key) and V, not K (d values per key).  The cache
// keeps K~ in fp16 with one power-of-two multiplier per key row, chosen from
// the row's own max |value| so that every row uses the top of the fp16 range
// (the same range rule the forward uses for Q rows); appending keys never
// touches earlier rows.  ("Sparse Projection Attention", Sec. 3.1.2 for the
// projection; the cache saving is the pages' argument for projected keys.)
//
// The cache rows themselves are written by the projection kernels (project.cu,
// output mode F16ROWS).
//
//   decode_kernel         one query per (batch, head) against keys 0 .. L-1,
//                         split over key chunks: q~ = q P_h (fp32, in every
//                         CTA from L2), scores
//                         from the fp16 cache in fp32, chunk max and sum, and
//                         the chunk's P V in fp32; writes (max, sum, O) per
//                         chunk.  HBM-bound: per key 2m + 4 bytes of cache and
//                         2 d_v bytes of V.
//   decode_combine_kernel the log-sum-exp merge of the chunks of one
//                         (batch, head) into the output row.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "kernels.cuh"

namespace spa {
namespace {

// ------------------------------------------------------------ decode
constexpr int kDecodeThreads = 256;

// grid (nsplit, BH), 256 threads.  Chunk c covers keys [c*chunk, min(L, (c+1)*chunk)).
template <int DV>
__global__ void __launch_bounds__(kDecodeThreads) decode_kernel(const DecodeParams p) {
  extern __shared__ float sc[];  // scores, then probabilities, of this chunk
  __shared__ float qs[128];      // q~ * log2(e)/sqrt(m)
  __shared__ float qpart[kDecodeThreads];
  __shared__ float red[kDecodeThreads / 32];
  __shared__ float oacc[kDecodeThreads / 32][DV];
  const int bh = blockIdx.y, split = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int k0 = split * p.chunk, n = min(p.L, k0 + p.chunk) - k0;

  // q~ = q P_h * log2(e)/sqrt(m), by every CTA of the (batch, head) (8 KB of
  // P_h from L2 at m = 32; a separate launch cost more than the work): thread
  // t sums column t % m over the rows l = t / m (mod G), coalesced across the
  // columns, and the G partial sums meet in shared memory
  {
    const int G = kDecodeThreads / p.m;  // row groups (m divides 256)
    const int k = tid % p.m, g = tid / p.m;
    const __nv_bfloat16* q = p.q + static_cast<size_t>(bh) * p.d;
    const __nv_bfloat16* P = p.P + static_cast<size_t>(bh % p.H) * p.d * p.m + k;
    float acc = 0.f;
#pragma unroll 4
    for (int l = g; l < p.d; l += G) acc = fmaf(__bfloat162float(q[l]), __bfloat162float(P[l * p.m]), acc);
    qpart[tid] = acc;
    __syncthreads();
    if (tid < p.m) {
      float s = 0.f;
      for (int gg = 0; gg < G; ++gg) s += qpart[gg * p.m + tid];
      qs[tid] = s * p.qscale;
    }
    __syncthreads();
  }

  // scores in log2 units: one key row per thread, m fp16 values in 16-byte pieces
  const uint16_t* kc = p.kc + (static_cast<size_t>(bh) * p.cap + k0) * p.m;
  const float* kmul = p.kc_mul + static_cast<size_t>(bh) * p.cap + k0;
  float tmax = -INFINITY;
  for (int j = tid; j < n; j += kDecodeThreads) {
    const uint4* row = reinterpret_cast<const uint4*>(kc + static_cast<size_t>(j) * p.m);
    float s = 0.f;
    for (int c = 0; c < p.m / 8; ++c) {
      const uint4 w = __ldg(row + c);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&ws[i]));
        s = fmaf(f.x, qs[8 * c + 2 * i], s);
        s = fmaf(f.y, qs[8 * c + 2 * i + 1], s);
      }
    }
    s *= __ldg(kmul + j);
    sc[j] = s;
    tmax = fmaxf(tmax, s);
  }
  // chunk max
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
  if (lane == 0) red[warp] = tmax;
  __syncthreads();
  float cmax = red[0];
#pragma unroll
  for (int w = 1; w < kDecodeThreads / 32; ++w) cmax = fmaxf(cmax, red[w]);
  __syncthreads();  // red is reused for the sum
  // probabilities and their sum
  float lsum = 0.f;
  for (int j = tid; j < n; j += kDecodeThreads) {
    const float e = exp2f(sc[j] - cmax);
    sc[j] = e;
    lsum += e;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
  if (lane == 0) red[warp] = lsum;
  __syncthreads();  // also publishes sc[]

  // O = sum_j p_j V_j: warp w takes keys w, w+8, ...; lane covers DV/32 columns
  constexpr int kCols = DV / 32;  // 2 or 4 bf16 per lane (4 or 8 bytes)
  const __nv_bfloat16* v = p.v + (static_cast<size_t>(bh) * p.cap + k0) * DV + lane * kCols;
  float o[kCols];
#pragma unroll
  for (int c = 0; c < kCols; ++c) o[c] = 0.f;
  int j = warp;
  for (; j + 3 * (kDecodeThreads / 32) < n; j += 4 * (kDecodeThreads / 32)) {
    float pj[4];
    float vv[4][kCols];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int jj = j + u * (kDecodeThreads / 32);
      pj[u] = sc[jj];
      const __nv_bfloat16* vr = v + static_cast<size_t>(jj) * DV;
      if constexpr (kCols == 4) {
        const uint2 w = __ldg(reinterpret_cast<const uint2*>(vr));
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.y));
        vv[u][0] = a.x; vv[u][1] = a.y; vv[u][2] = b.x; vv[u][3] = b.y;
      } else {
        const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(vr));
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
        vv[u][0] = a.x; vv[u][1] = a.y;
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int c = 0; c < kCols; ++c) o[c] = fmaf(pj[u], vv[u][c], o[c]);
  }
  for (; j < n; j += kDecodeThreads / 32) {
    const float pj = sc[j];
    const __nv_bfloat16* vr = v + static_cast<size_t>(j) * DV;
#pragma unroll
    for (int c = 0; c < kCols; ++c) o[c] = fmaf(pj, __bfloat162float(vr[c]), o[c]);
  }
#pragma unroll
  for (int c = 0; c < kCols; ++c) oacc[warp][lane * kCols + c] = o[c];
  __syncthreads();
  // chunk result: (max, sum, O[DV]) in log2 units
  float* part = p.part + (static_cast<size_t>(bh) * p.nsplit + split) * (2 + DV);
  if (tid < DV) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kDecodeThreads / 32; ++w) s += oacc[w][tid];
    part[2 + tid] = s;
  }
  if (tid == 0) {
    float l = 0.f;
#pragma unroll
    for (int w = 0; w < kDecodeThreads / 32; ++w) l += red[w];
    part[0] = cmax;
    part[1] = l;
  }
}

// grid BH, 256 threads: out = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c.
// The chunk maxima are reduced by the whole block; then 256 / DV groups of
// DV threads (one per output column) take every (256 / DV)-th chunk, with the
// loads of several chunks in flight, and meet in shared memory.
template <int DV>
__global__ void __launch_bounds__(kDecodeThreads) decode_combine_kernel(const DecodeParams p) {
  constexpr int G = kDecodeThreads / DV;
  __shared__ float red[kDecodeThreads / 32];
  __shared__ float acc_o[G][DV], acc_l[G];
  const int bh = blockIdx.x, tid = threadIdx.x, c = tid % DV, g = tid / DV;
  const float* part = p.part + static_cast<size_t>(bh) * p.nsplit * (2 + DV);
  float M = -INFINITY;
  for (int s = tid; s < p.nsplit; s += kDecodeThreads) M = fmaxf(M, part[s * (2 + DV)]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if ((tid & 31) == 0) red[tid >> 5] = M;
  __syncthreads();
  M = red[0];
#pragma unroll
  for (int w = 1; w < kDecodeThreads / 32; ++w) M = fmaxf(M, red[w]);
  float l = 0.f, o = 0.f;
#pragma unroll 4
  for (int s = g; s < p.nsplit; s += G) {
    const float* ps = part + s * (2 + DV);
    const float w = exp2f(ps[0] - M);
    l = fmaf(w, ps[1], l);
    o = fmaf(w, ps[2 + c], o);
  }
  acc_o[g][c] = o;
  if (c == 0) acc_l[g] = l;
  __syncthreads();
  if (g == 0) {
    float os = 0.f, ls = 0.f;
#pragma unroll
    for (int gg = 0; gg < G; ++gg) {
      os += acc_o[gg][c];
      ls += acc_l[gg];
    }
    p.out[static_cast<size_t>(bh) * DV + c] = os / ls;
  }
}

}  // namespace

void decode_split(int BH, int L, int sms, int* nsplit, int* chunk) {
  // about eight CTAs' worth of key chunks per SM, each a multiple of 32 keys
  // and at most kDecodeMaxChunk (its scores stay in shared memory)
  const long long want = (8LL * sms + BH - 1) / BH;
  int ns = static_cast<int>(want < 1 ? 1 : want);
  const int by_len = (L + 255) / 256;  // at least 256 keys per chunk
  if (ns > by_len) ns = by_len;
  const int min_ns = (L + kDecodeMaxChunk - 1) / kDecodeMaxChunk;
  if (ns < min_ns) ns = min_ns;
  int ch = (L + ns - 1) / ns;
  ch = (ch + 31) / 32 * 32;
  *chunk = ch;
  *nsplit = (L + ch - 1) / ch;
}

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(p.chunk) * sizeof(float);
  dim3 grid(p.nsplit, p.BH);
  cudaError_t e;
  if (p.dv == 128) {
    e = cudaFuncSetAttribute(decode_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    decode_kernel<128><<<grid, kDecodeThreads, smem, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    decode_combine_kernel<128><<<p.BH, kDecodeThreads, 0, stream>>>(p);
  } else if (p.dv == 64) {
    e = cudaFuncSetAttribute(decode_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    decode_kernel<64><<<grid, kDecodeThreads, smem, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    decode_combine_kernel<64><<<p.BH, kDecodeThreads, 0, stream>>>(p);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace spa
