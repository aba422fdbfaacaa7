// attn_f32.cu -- the fp32 path: scores, mask, online softmax and the value
// product in true fp32 FMA arithmetic (no TF32, no reduced-precision
// operands), for fp32 inputs that want fp32-level agreement.
//
// One warp owns one query row.  Keys are taken 32 at a time, one per lane:
// each lane forms its score <qp_i, kp_j> / sqrt(m), the warp takes the chunk
// max, rescales its running output and sum by exp(m_old - m_new) and adds
// exp(s_j - m_new) * v_j, broadcasting each lane's weight with a shuffle.
// This is the streaming (online) softmax, so no N x N matrix is formed
// ("Scaling Attention via Feature Sparsity", FlashSFA description: tiling and
// online softmax; the result equals the row softmax of SPA Algorithm 1 step 5).
#include <math.h>

#include "kernels.cuh"

namespace spa {
namespace {

constexpr int kWarps = 4;

template <int DVMAX>
__global__ void __launch_bounds__(kWarps * 32) attn_f32_kernel(const AttnF32Params p) {
  __shared__ float qs[kWarps][128];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows_per_bh = (p.N + kWarps - 1) / kWarps;
  const int bh = blockIdx.x / rows_per_bh;
  const int i = (blockIdx.x % rows_per_bh) * kWarps + warp;
  if (i >= p.N) return;  // whole warp leaves together; no block barrier below

  const size_t qk_off = static_cast<size_t>(bh) * p.N * p.m;
  const float* Kp = p.Kp + qk_off;
  const float* V = p.V + static_cast<size_t>(bh) * p.N * p.dv;
  for (int c = lane; c < p.m; c += 32) qs[warp][c] = p.Qp[qk_off + static_cast<size_t>(i) * p.m + c];
  __syncwarp();

  constexpr int NC = DVMAX / 32;
  float o[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c) o[c] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;
  const int nkeys = p.causal ? i + 1 : p.N;

  for (int j0 = 0; j0 < nkeys; j0 += 32) {
    const int j = j0 + lane;
    float s = -INFINITY;
    if (j < nkeys) {
      const float* kr = Kp + static_cast<size_t>(j) * p.m;
      float acc = 0.f;
      for (int c = 0; c < p.m; ++c) acc = fmaf(qs[warp][c], kr[c], acc);
      s = acc * p.scale;
    }
    float cmax = s;
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, o2));
    const float m_new = fmaxf(m_run, cmax);
    const float alpha = expf(m_run - m_new);  // 0 on the first chunk
    const float pj = (j < nkeys) ? expf(s - m_new) : 0.f;
    float psum = pj;
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o2);
    l_run = l_run * alpha + psum;
    m_run = m_new;
#pragma unroll
    for (int c = 0; c < NC; ++c) o[c] *= alpha;
    const int tmax = min(32, nkeys - j0);
    for (int t = 0; t < tmax; ++t) {
      const float pt = __shfl_sync(0xffffffffu, pj, t);
      const float* vr = V + static_cast<size_t>(j0 + t) * p.dv;
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        const int col = lane + 32 * c;
        if (col < p.dv) o[c] = fmaf(pt, vr[col], o[c]);
      }
    }
  }
  float* dst = p.out + (static_cast<size_t>(bh) * p.N + i) * p.dv;
  const float inv = 1.f / l_run;
  if (p.lse != nullptr && lane == 0) p.lse[static_cast<size_t>(bh) * p.N + i] = m_run + logf(l_run);
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const int col = lane + 32 * c;
    if (col < p.dv) dst[col] = o[c] * inv;
  }
}

}  // namespace

cudaError_t launch_attn_f32(const AttnF32Params& p, cudaStream_t stream) {
  const long long rows_per_bh = (p.N + kWarps - 1) / kWarps;
  const long long blocks = rows_per_bh * p.BH;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  dim3 grid(static_cast<unsigned>(blocks));
  if (p.dv <= 64) attn_f32_kernel<64><<<grid, kWarps * 32, 0, stream>>>(p);
  else if (p.dv <= 128) attn_f32_kernel<128><<<grid, kWarps * 32, 0, stream>>>(p);
  else attn_f32_kernel<256><<<grid, kWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace spa
