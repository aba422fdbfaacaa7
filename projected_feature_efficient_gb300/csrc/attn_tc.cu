// attn_tc.cu -- fused projected-feature attention on the 5th-generation tensor
// cores (tcgen05) for bf16 inputs.
//
// Per CTA: one tile of 128 query rows of one (batch, head); thread r owns
// query row r, which is also TMEM lane r of every accumulator.  For each tile
// of 128 keys:
//   1. the score-operand tile of Kp (pre-converted by the projection kernel
//      into the tensor cores' interleaved layout) arrives with one bulk copy,
//      the V tile with two/one TMA tensor copies (128-byte swizzle);
//   2. S = Qp Kp^T accumulates in TMEM (fp32), K-depth KD = m or 3m;
//   3. each thread reads its S row, multiplies by its row and tile range
//      factors (which carry log2(e)/sqrt(m)), masks, and runs the online
//      softmax in base 2: running max, exp2, running sum, and -- when the
//      max moved -- rescales its O row in TMEM;
//   4. the probabilities, rounded to bf16, are written back into the S
//      columns of TMEM and O += P V runs with P read straight from TMEM;
//   5. after the last key tile, O / l goes to global memory in fp32.
// The N x N matrix never leaves TMEM ("Projection-Decomposition Attention",
// Sec. 4.2: S~ can be streamed; "Scaling Attention via Feature Sparsity",
// FlashSFA: tiling plus online softmax).  Under a causal mask only key tiles
// at or left of the diagonal are visited and only the diagonal tile is masked.
#include <math.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace spa {
namespace {

using namespace ptx;

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait

__device__ __forceinline__ uint8_t* align1k(uint8_t* p) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return reinterpret_cast<uint8_t*>((a + 1023) & ~static_cast<uintptr_t>(1023));
}

template <int KD, int DV>
struct SmemPlan {
  static constexpr int kTileBytes = kTileRows * KD * 2;
  static constexpr int kQ = 0;
  static constexpr int kK = kTileBytes;
  static constexpr int kV = 2 * kTileBytes;            // multiple of 1024: KD % 16 == 0
  static constexpr int kBytes = kV + DV * kTileRows * 2;
  // at most two CTAs per SM so that two TMEM allocations of 256 columns fit
  static constexpr int kLaunch = (kBytes + 1024) > 100 * 1024 ? kBytes + 1024 : 100 * 1024;
};

template <int KD, int DV, bool F16OPS>
__global__ void __launch_bounds__(128, 1) attn_tc_kernel(const AttnTcParams p,
                                                         const __grid_constant__ CUtensorMap vmap) {
  using Plan = SmemPlan<KD, DV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1k(smem_raw);
  uint8_t* sQ = smem + Plan::kQ;
  uint8_t* sK = smem + Plan::kK;
  uint8_t* sV = smem + Plan::kV;
  __shared__ uint64_t bar_load, bar_mma;
  __shared__ uint32_t tmem_base_sh;

  const int tid = threadIdx.x, warp = tid >> 5;
  const int NT = p.NT;
  const int bh = blockIdx.x / NT;
  const int qt = NT - 1 - static_cast<int>(blockIdx.x % NT);  // longest causal rows first

  constexpr uint32_t kCols = 256;  // S/P: columns [0,128); O: [128, 128+DV)
  if (warp == 0) {
    tmem_alloc(&tmem_base_sh, kCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bar_load, 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
    prefetch_tmap(&vmap);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tmem_base_sh;
  const uint32_t t_lane = tb + (static_cast<uint32_t>(warp * 32) << 16);
  const uint32_t tS = tb, tO = tb + 128;  // S/P and O accumulators

  constexpr uint32_t kIdescS = idesc_f16(128, 128, F16OPS ? kFmtF16 : kFmtBF16, 0, 0);
  constexpr uint32_t kIdescPV = idesc_f16(128, DV, kFmtBF16, 0, 1);
  constexpr int kTileElems = kTileRows * KD;

  const int row = qt * kTileRows + tid;
  const float qm = p.qmul[static_cast<size_t>(bh) * NT * kTileRows + row];
  const float* kmul = p.kmul + static_cast<size_t>(bh) * NT;
  const uint16_t* Ks = p.Ks + static_cast<size_t>(bh) * NT * kTileElems;
  const int nkv = p.causal ? qt + 1 : NT;

  float m_run = -INFINITY, l_run = 0.f;
  uint32_t ph_load = 0, ph_mma = 0;
  bool ok = true;
  uint64_t* pending = nullptr;  // barrier of the wait that gave up
  uint32_t pending_ph = 0;

  for (int j = 0; j < nkv; ++j) {
    if (tid == 0) {
      uint32_t bytes = Plan::kTileBytes + DV * kTileRows * 2 + (j == 0 ? Plan::kTileBytes : 0);
      mbar_arrive_expect_tx(&bar_load, bytes);
      if (j == 0)
        bulk_g2s(sQ, p.Qs + (static_cast<size_t>(bh) * NT + qt) * kTileElems, Plan::kTileBytes,
                 &bar_load);
      bulk_g2s(sK, Ks + static_cast<size_t>(j) * kTileElems, Plan::kTileBytes, &bar_load);
#pragma unroll
      for (int h = 0; h < DV / 64; ++h)
        tma_load_3d(sV + h * 16384, &vmap, h * 64, j * kTileRows, bh, &bar_load);
    }
    ok = __syncthreads_and(mbar_wait(&bar_load, ph_load, kWaitLimitNs));
    if (!ok) { pending = &bar_load; pending_ph = ph_load; break; }
    ph_load ^= 1;

    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int s = 0; s < KD / 16; ++s)
        mma_ss(tS, smem_desc(smem_u32(sQ) + s * 4096, 2048, 128, kLayoutInterleave),
               smem_desc(smem_u32(sK) + s * 4096, 2048, 128, kLayoutInterleave), kIdescS, s > 0);
      mma_commit(&bar_mma);
    }
    ok = __syncthreads_and(mbar_wait(&bar_mma, ph_mma, kWaitLimitNs));
    if (!ok) { pending = &bar_mma; pending_ph = ph_mma; break; }
    ph_mma ^= 1;
    tc_fence_after();

    // ---- online softmax on row `row`, base-2 logits
    float x[128];
#pragma unroll
    for (int c0 = 0; c0 < 128; c0 += 32) {
      uint32_t r[32];
      tmem_ld32(t_lane + c0, r);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) x[c0 + i] = __uint_as_float(r[i]);
    }
    const float mult = qm * kmul[j];
    int kvalid = p.N - j * kTileRows;                 // keys of this tile inside N
    if (p.causal && j == qt) kvalid = min(kvalid, tid + 1);
    float tmax = -INFINITY;
#pragma unroll
    for (int c = 0; c < 128; ++c) {
      x[c] = c < kvalid ? x[c] * mult : -INFINITY;
      tmax = fmaxf(tmax, x[c]);
    }
    const float m_new = fmaxf(m_run, tmax);
    const float alpha = ex2(m_run - m_new);
    float lsum = 0.f;
#pragma unroll
    for (int c = 0; c < 128; ++c) {
      x[c] = ex2(x[c] - m_new);
      lsum += x[c];
    }
    l_run = l_run * alpha + lsum;
    m_run = m_new;

    if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {  // O row *= alpha
#pragma unroll
      for (int c0 = 0; c0 < DV; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(t_lane + 128 + c0, r);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
        tmem_st32(t_lane + 128 + c0, r);
      }
    }
    {  // P (bf16 pairs) into S columns [0, 64)
      uint32_t r[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) r[i] = pack_bf16x2(x[2 * i], x[2 * i + 1]);
      tmem_st32(t_lane, r);
#pragma unroll
      for (int i = 0; i < 32; ++i) r[i] = pack_bf16x2(x[64 + 2 * i], x[64 + 2 * i + 1]);
      tmem_st32(t_lane + 32, r);
    }
    tmem_wait_st();
    tc_fence_before();
    __syncthreads();

    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int s = 0; s < 8; ++s)
        mma_ts(tO, tS + s * 8,
               smem_desc(smem_u32(sV) + s * 2048, 16384, 1024, kLayoutSwizzle128), kIdescPV,
               (j > 0 || s > 0) ? 1u : 0u);
      mma_commit(&bar_mma);
    }
    ok = __syncthreads_and(mbar_wait(&bar_mma, ph_mma, kWaitLimitNs));
    if (!ok) { pending = &bar_mma; pending_ph = ph_mma; break; }
    ph_mma ^= 1;
  }

  if (ok) {
    tc_fence_after();
    const float inv = 1.f / l_run;
    float* dst = p.out + (static_cast<size_t>(bh) * p.N + row) * DV;
#pragma unroll
    for (int c0 = 0; c0 < DV; c0 += 32) {
      uint32_t r[32];
      tmem_ld32(t_lane + 128 + c0, r);
      tmem_wait_ld();
      if (row < p.N) {
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          float4 v4 = make_float4(__uint_as_float(r[i]) * inv, __uint_as_float(r[i + 1]) * inv,
                                  __uint_as_float(r[i + 2]) * inv, __uint_as_float(r[i + 3]) * inv);
          *reinterpret_cast<float4*>(dst + c0 + i) = v4;
        }
      }
    }
  } else {
    if (tid == 0) atomicExch(p.err, 1);
    // let copies / MMAs still in flight land before the CTA's memory is reused
    mbar_wait(pending, pending_ph, kWaitLimitNs);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, kCols);
}

template <int KD, int DV, bool F16OPS>
cudaError_t launch_tc(const AttnTcParams& p, cudaStream_t stream) {
  using Plan = SmemPlan<KD, DV>;
  auto kern = attn_tc_kernel<KD, DV, F16OPS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Plan::kLaunch);
  if (e != cudaSuccess) return e;
  const long long blocks = static_cast<long long>(p.NT) * p.BH;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  kern<<<static_cast<unsigned>(blocks), 128, Plan::kLaunch, stream>>>(p, p.vmap);
  return cudaGetLastError();
}

template <int DV>
cudaError_t launch_dv(const AttnTcParams& p, cudaStream_t stream) {
  if (!p.f16_ops) {
    if (p.KD == 48) return launch_tc<48, DV, false>(p, stream);
    return cudaErrorInvalidValue;
  }
  switch (p.KD) {
    case 32: return launch_tc<32, DV, true>(p, stream);
    case 64: return launch_tc<64, DV, true>(p, stream);
    case 128: return launch_tc<128, DV, true>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_attn_tc(const AttnTcParams& p, cudaStream_t stream) {
  if (p.dv == 64) return launch_dv<64>(p, stream);
  if (p.dv == 128) return launch_dv<128>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace spa
