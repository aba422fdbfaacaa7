// bwd_finish.cu -- the last step of the fused backward: the gradients of the
// projection (SPA paper, Sec. 3.1.2: Qp = Q P_h, Kp = K P_h), given the
// gradients dQp (the fused kernel's fp32 accumulator) and dKp (its bf16 hi | lo
// rows):
//   dq = dQp P_h^T,   dk = dKp P_h^T             (fp32 rows [BH][N][d])
//   dP_h = sum_b ( q_b,h^T dQp + k_b,h^T dKp )    (fp32 [H][d][m])
// in one pass over q, k and the two gradients, on the tensor cores, for m = 32
// and d = 128.
//
// A unit is one 128-row tile of one (side, b, h), side = q or k; units are
// ordered by head, then side, batch and tile, and each persistent CTA takes a
// contiguous range of them (two CTAs per SM).  Per unit:
//   - one thread loads the X tile (q or k, two 64-column boxes by TMA, 128-byte
//     swizzle) and the gradient tile G into shared memory: for k the dKp rows
//     by TMA (already bf16 hi | lo, 64 values = 128 bytes per row); for q the
//     raw fp32 dQp tile by one bulk copy, which every thread then splits in
//     place into bf16 hi | lo (its own row: 32 fp32 -> 64 bf16, both 128 bytes,
//     in the same 128-byte swizzle);
//   - the same thread issues   out = G [P_h | P_h]^T   (M = 128 rows, N = d,
//     K = 64; G and the duplicated P_h rows both K-major)  and
//     dPacc += X^T G   (M = d, N = 64, K = 128 rows; X^T and G read MN-major
//     from the same tiles), and commits;
//   - as soon as the products have read the tiles, the next unit's loads go
//     out, and all 128 threads move `out` from tensor memory through a
//     shared-memory staging tile to dq / dk with TMA stores (rows past N are
//     clipped).
// When the head changes (and at the end) the threads fold the accumulator's hi
// and lo halves (dP = R[:, :m] + R[:, m:]) and add it to dP_h with one bulk
// reduce-add; dP is zeroed before the launch.  Products accumulate in fp32;
// the gradients enter as bf16 hi + lo pairs (16 significant bits).
//
// Every wait is bounded; a CTA that gives up sets the device error word, lets
// its own copies and products finish, and frees its tensor memory.
#include <cuda_bf16.h>

#include "kernels.cuh"
#include "bwd_common.cuh"
#include "ptx.cuh"

namespace spa {
namespace {

using namespace ptx;

constexpr int kFinThreads = 128;
constexpr int kFinBox = kTileRows * 128;  // one 128-row x 128-byte tile / box: 16 KB

struct FinPlan {  // offsets from the 1024-byte-aligned base of dynamic shared memory
  static constexpr int kX = 0;               // X tile, two boxes [128][64] bf16
  static constexpr int kG = 2 * kFinBox;     // gradient tile [128][64] bf16 (raw dQp first, for q)
  static constexpr int kP2 = 3 * kFinBox;    // rows of [P_h | P_h], [128][64] bf16
  static constexpr int kOut = 4 * kFinBox;   // two output staging boxes [128][32] fp32
  static constexpr int kBytes = 6 * kFinBox;
  static constexpr int kLaunch = kBytes + 1024;
  static constexpr uint32_t kColsOut = 0, kColsDp = 128, kCols = 256;  // tensor memory
};

// One 16-byte chunk of shared memory, by shared-window address.
__device__ __forceinline__ void ld_shared_v4(uint32_t a, uint32_t (&v)[4]) {
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
               : "r"(a));
}

struct Unit {
  int h, side, bh, tile;
};

__global__ void __launch_bounds__(kFinThreads) bwd_finish_kernel(
    const BwdFinishParams p, const __grid_constant__ CUtensorMap qmap,
    const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap xkmap,
    const __grid_constant__ CUtensorMap dqmap, const __grid_constant__ CUtensorMap dkmap) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_full, bar_mma;
  __shared__ uint32_t tmem_base_sh;
  const int tid = threadIdx.x, warp = tid >> 5;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const long long per_head = 2LL * p.B * p.NT;
  const long long U = per_head * p.H;
  const long long G = gridDim.x;
  const long long u0 = blockIdx.x * U / G, u1 = (blockIdx.x + 1) * U / G;
  auto unit = [&](long long u) {
    Unit x;
    x.h = static_cast<int>(u / per_head);
    const long long r = u % per_head;
    x.side = static_cast<int>(r / (static_cast<long long>(p.B) * p.NT));
    const long long r2 = r % (static_cast<long long>(p.B) * p.NT);
    x.bh = static_cast<int>(r2 / p.NT) * p.H + x.h;
    x.tile = static_cast<int>(r2 % p.NT);
    return x;
  };
  int loads = 0, commits = 0;  // thread 0: unit loads started, MMA commits
  auto load = [&](long long u) {  // thread 0 only
    const Unit x = unit(u);
    ++loads;
    mbar_arrive_expect_tx(&bar_full, 3 * kFinBox);
    const CUtensorMap* xm = x.side == 0 ? &qmap : &kmap;
    tma_load_3d(smem_raw + (sbase - smem_u32(smem_raw)) + FinPlan::kX, xm, 0, x.tile * kTileRows,
                x.bh, &bar_full);
    tma_load_3d(smem_raw + (sbase - smem_u32(smem_raw)) + FinPlan::kX + kFinBox, xm, 64,
                x.tile * kTileRows, x.bh, &bar_full);
    uint8_t* g = smem_raw + (sbase - smem_u32(smem_raw)) + FinPlan::kG;
    if (x.side == 0)
      bulk_g2s(g, p.dqacc + (static_cast<size_t>(x.bh) * p.NT + x.tile) * kTileRows * 32, kFinBox,
               &bar_full);
    else
      tma_load_3d(g, &xkmap, 0, x.tile * kTileRows, x.bh, &bar_full);
  };

  if (warp == 0) {
    tmem_alloc(&tmem_base_sh, FinPlan::kCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    prefetch_tmap(&qmap);
    prefetch_tmap(&kmap);
    prefetch_tmap(&xkmap);
    prefetch_tmap(&dqmap);
    prefetch_tmap(&dkmap);
    mbar_init(&bar_full, 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
    if (u0 < u1) load(u0);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tmem_base_sh;
  const uint32_t lane_base = tb + (static_cast<uint32_t>(warp * 32) << 16);
  const int r = tid;  // row of the tile (TMEM lane) / row of d (dP accumulator lane)
  const uint32_t sw = static_cast<uint32_t>(r & 7);

  // fold the dP accumulator of head h and add it to dP_h (one bulk reduce-add)
  auto flush = [&](int h) {
    tc_fence_after();
    uint32_t v0[32], v1[32];
    tmem_ld32(lane_base + FinPlan::kColsDp, v0);
    tmem_ld32(lane_base + FinPlan::kColsDp + 32, v1);
    tmem_wait_ld();
    if (tid == 0) bulk_wait_group_read<0>();  // the staging tile is no longer read
    __syncthreads();
    const uint32_t row = sbase + FinPlan::kOut + r * 128;
#pragma unroll
    for (int c = 0; c < 8; ++c)
      st_shared_v4(row + c * 16,
                   __float_as_uint(__uint_as_float(v0[4 * c]) + __uint_as_float(v1[4 * c])),
                   __float_as_uint(__uint_as_float(v0[4 * c + 1]) + __uint_as_float(v1[4 * c + 1])),
                   __float_as_uint(__uint_as_float(v0[4 * c + 2]) + __uint_as_float(v1[4 * c + 2])),
                   __float_as_uint(__uint_as_float(v0[4 * c + 3]) + __uint_as_float(v1[4 * c + 3])));
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      bulk_reduce_add_f32(p.dP + static_cast<size_t>(h) * p.d * p.m, sbase + FinPlan::kOut,
                          kFinBox);
      bulk_commit_group();
      bulk_wait_group_read<0>();
    }
  };

  bool ok = true;
  int staged_h = -1;
  bool dp_fresh = true;  // the next dP product starts the head's accumulator
  for (long long u = u0; ok && u < u1; ++u) {
    const int i = static_cast<int>(u - u0);
    const Unit x = unit(u);
    if (x.h != staged_h) {
      if (staged_h >= 0) flush(staged_h);
      // rows of [P_h | P_h]: row l = P_h[l][0..31] twice, 128-byte swizzle
      const uint4* src = reinterpret_cast<const uint4*>(p.P + (static_cast<size_t>(x.h) * p.d + r) * 32);
      uint4 pv[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) pv[c] = __ldg(src + c);
      const uint32_t row = sbase + FinPlan::kP2 + r * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        st_shared_v4(row + ((c ^ sw) << 4), pv[c & 3].x, pv[c & 3].y, pv[c & 3].z, pv[c & 3].w);
      staged_h = x.h;
      dp_fresh = true;
    }
    ok = __syncthreads_and(mbar_wait(&bar_full, i & 1, p.limit_ns));
    if (!ok) break;
    if (x.side == 0) {  // raw fp32 dQp row -> bf16 hi | lo row, in place
      const uint32_t row = sbase + FinPlan::kG + r * 128;
      uint32_t v[32];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t t[4];
        ld_shared_v4(row + ((c ^ sw) << 4), t);
        v[4 * c] = t[0];
        v[4 * c + 1] = t[1];
        v[4 * c + 2] = t[2];
        v[4 * c + 3] = t[3];
      }
      uint32_t hi[16], lo[16];
#pragma unroll
      for (int j = 0; j < 16; ++j)
        split_pair(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]), hi[j], lo[j]);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        st_shared_v4(row + ((c ^ sw) << 4), hi[4 * c], hi[4 * c + 1], hi[4 * c + 2], hi[4 * c + 3]);
        st_shared_v4(row + (((c + 4) ^ sw) << 4), lo[4 * c], lo[4 * c + 1], lo[4 * c + 2],
                     lo[4 * c + 3]);
      }
    }
    // the P rows and the converted gradient rows are visible to the tensor
    // cores; the previous unit's reads of tensor memory are done
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      constexpr uint32_t kIdOut = idesc_f16(128, 128, kFmtBF16, 0, 0);
      constexpr uint32_t kIdDp = idesc_f16(128, 64, kFmtBF16, 1, 1);
      const uint32_t sG = sbase + FinPlan::kG, sP = sbase + FinPlan::kP2, sX = sbase + FinPlan::kX;
#pragma unroll
      for (int k = 0; k < 4; ++k)  // out = G [P | P]^T: K = 64 (hi, lo) in four steps
        mma_ss(tb + FinPlan::kColsOut, smem_desc(sG + k * 32, 16, 1024, kLayoutSwizzle128),
               smem_desc(sP + k * 32, 16, 1024, kLayoutSwizzle128), kIdOut, k > 0);
#pragma unroll
      for (int k = 0; k < 8; ++k)  // dPacc += X^T G: K = 128 rows in eight steps
        mma_ss(tb + FinPlan::kColsDp, smem_desc(sX + k * 2048, kFinBox, 1024, kLayoutSwizzle128),
               smem_desc(sG + k * 2048, kFinBox, 1024, kLayoutSwizzle128), kIdDp,
               (dp_fresh && k == 0) ? 0u : 1u);
      mma_commit(&bar_mma);
      ++commits;
    }
    dp_fresh = false;
    ok = __syncthreads_and(mbar_wait(&bar_mma, i & 1, p.limit_ns));
    if (!ok) break;
    // the products have read X and G: the next unit's tiles may come in
    if (tid == 0 && u + 1 < u1) load(u + 1);
    tc_fence_after();
    // ---- out (fp32) -> dq / dk through two staging boxes and TMA stores
    const CUtensorMap* om = x.side == 0 ? &dqmap : &dkmap;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      uint32_t v[32];
      tmem_ld32(lane_base + FinPlan::kColsOut + b * 32, v);
      tmem_wait_ld();
      const uint32_t box = sbase + FinPlan::kOut + (b & 1) * kFinBox;
      if (tid == 0) bulk_wait_group_read<1>();  // this box's previous store has read it
      __syncthreads();
      const uint32_t row = box + r * 128;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        st_shared_v4(row + ((q ^ sw) << 4), v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      fence_proxy_async_smem();
      __syncthreads();
      if (tid == 0) {
        tma_store_3d(om, box, b * 32, x.tile * kTileRows, x.bh);
        bulk_commit_group();
      }
    }
  }
  if (ok && staged_h >= 0) flush(staged_h);
  if (tid == 0) {
    if (!ok) {
      atomicExch(p.err, 1);
      mma_commit(&bar_mma);  // a product may still be in flight
      mbar_wait(&bar_mma, commits & 1, p.limit_ns);
    }
    // the last tile load started has landed (all of them have, unless a wait gave up)
    if (loads > 0) mbar_wait(&bar_full, (loads - 1) & 1, p.limit_ns);
    bulk_wait_group_read<0>();  // the stores and the reduce-add have read shared memory
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, FinPlan::kCols);
}

}  // namespace

bool bwd_finish_tc_supported(int d, int m) { return d == 128 && m == 32; }

cudaError_t launch_bwd_finish_tc(const BwdFinishParams& p, cudaStream_t stream) {
  if (!bwd_finish_tc_supported(p.d, p.m)) return cudaErrorInvalidValue;
  cudaError_t e = cudaMemsetAsync(p.dP, 0, static_cast<size_t>(p.H) * p.d * p.m * sizeof(float),
                                  stream);
  if (e != cudaSuccess) return e;
  const long long units = 2LL * p.B * p.H * p.NT;
  if (units == 0) return cudaSuccess;
  e = cudaFuncSetAttribute(bwd_finish_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           FinPlan::kLaunch);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  // two CTAs per SM: 2 x 256 tensor-memory columns, 2 x 97 KB of shared memory
  const long long grid = units < 2LL * sms ? units : 2LL * sms;
  bwd_finish_kernel<<<static_cast<unsigned>(grid), kFinThreads, FinPlan::kLaunch, stream>>>(
      p, p.qmap, p.kmap, p.xkmap, p.dqmap, p.dkmap);
  return cudaGetLastError();
}

}  // namespace spa
