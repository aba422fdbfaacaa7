// bwd_finish.cu -- the last step of the fused backward: the gradients of the
// projection (SPA paper, Sec. 3.1.2: Qp = Q P_h, Kp = K P_h; Sec. 3.4.1: the
// gradient flows to Q and to the projection through Qp), given the fp32
// gradients dQp and dKp the fused kernel left in its accumulators:
//   dq = dQp P_h^T,   dk = dKp P_h^T             (fp32 rows [BH][N][d])
//   dP_h = sum_b ( q_b,h^T dQp + k_b,h^T dKp )    (fp32 [H][d][m])
// in one pass over q, k and the two gradients, on the tensor cores, for
// d in {64, 128} and m in {16, 32, 64}.
//
// A unit is one 128-row tile of one (side, b, h), side = q or k; units are
// ordered by head, then side, batch and tile, and each persistent CTA takes a
// contiguous range of them.  Per unit:
//   - one thread loads the X tile (q or k: d/64 boxes of 64 columns by TMA,
//     128-byte swizzle) and the raw fp32 gradient tile (one bulk copy of the
//     accumulator's tile, laid out in slabs as bwd_common.cuh states);
//   - every thread reads its row of the raw tile and, once all have read,
//     writes it back in place as bf16 hi | lo (hi = bf16(v), lo = bf16(v - hi),
//     16 significant bits) in the 128-byte swizzle, G = [hi | lo], padded with
//     zeros to whole 128-byte rows (m = 16);
//   - one thread issues   out = G [P_h | P_h | 0]^T   (M = 128 rows, N = d,
//     K = the padded width; both K-major)  and  dPacc += X^T G  (M = 128
//     features, N = the padded width, K = 128 rows; both read MN-major from
//     the same tiles; at d = 64 the second 64 features are a zero box), and
//     commits;
//   - as soon as the products have read the tiles, the next unit's loads go
//     out, and all 128 threads move `out` from tensor memory through a
//     shared-memory staging tile to dq / dk with TMA stores (rows past N are
//     clipped).
// When the head changes (and at the end) the threads fold the accumulator's hi
// and lo halves (dP = R[:, :m] + R[:, m:m+m]) and add it to dP_h with one bulk
// reduce-add; dP is zeroed before the launch.  Products accumulate in fp32.
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

template <int D, int M>
struct FinPlan {  // offsets from the 1024-byte-aligned base of dynamic shared memory
  static constexpr int kGW = 2 * M;                 // hi | lo values per gradient row
  static constexpr int kGWP = kGW < 64 ? 64 : kGW;  // padded to whole 128-byte rows
  static constexpr int kGB = kGWP / 64;             // 128-byte boxes per G / P2 row
  static constexpr int kX = 0;                      // X tile, two boxes [128][64] bf16
  static constexpr int kG = 2 * kFinBox;            // G tile (the raw fp32 tile first)
  static constexpr int kP2 = kG + kGB * kFinBox;    // rows of [P_h | P_h | 0]
  static constexpr int kOut = kP2 + kGB * kFinBox;  // two output staging boxes [128][32] fp32
  static constexpr int kBytes = kOut + 2 * kFinBox;
  static constexpr int kLaunch = kBytes + 1024;
  static constexpr int kRawBytes = kTileRows * M * 4;
  static constexpr int kSlab = dq_slab_cols(M);     // accumulator slab width (columns)
  static constexpr uint32_t kColsOut = 0, kColsDp = 128, kCols = 256;  // tensor memory
  static_assert(kRawBytes <= kGB * kFinBox, "raw gradient tile does not fit the G tile");
  static_assert(D * M * 4 <= 2 * kFinBox, "dP staging does not fit");
  static_assert(D == 64 || D == 128, "d must be 64 or 128");
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

template <int D, int M>
__global__ void __launch_bounds__(kFinThreads, 1) bwd_finish_kernel(
    const BwdFinishParams p, const __grid_constant__ CUtensorMap qmap,
    const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap dqmap,
    const __grid_constant__ CUtensorMap dkmap) {
  using Plan = FinPlan<D, M>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_full, bar_mma;
  __shared__ uint32_t tmem_base_sh;
  const int tid = threadIdx.x, warp = tid >> 5;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - smem_u32(smem_raw));
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
    mbar_arrive_expect_tx(&bar_full, D / 64 * kFinBox + Plan::kRawBytes);
    const CUtensorMap* xm = x.side == 0 ? &qmap : &kmap;
#pragma unroll
    for (int b = 0; b < D / 64; ++b)
      tma_load_3d(smem + Plan::kX + b * kFinBox, xm, 64 * b, x.tile * kTileRows, x.bh, &bar_full);
    const float* acc = x.side == 0 ? p.dqacc : p.dkacc;
    bulk_g2s(smem + Plan::kG, acc + (static_cast<size_t>(x.bh) * p.NT + x.tile) * kTileRows * M,
             Plan::kRawBytes, &bar_full);
  };

  if (warp == 0) {
    tmem_alloc(&tmem_base_sh, Plan::kCols);
    tmem_relinquish();
  }
  if (D == 64) {  // the X tile's second box stays zero: features 64..127 of X^T
    const uint32_t z = sbase + Plan::kX + kFinBox + tid * 128;
#pragma unroll
    for (int c = 0; c < 8; ++c) st_shared_v4(z + c * 16, 0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
  }
  if (tid == 0) {
    prefetch_tmap(&qmap);
    prefetch_tmap(&kmap);
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
  const int r = tid;  // row of the tile (TMEM lane) / feature row of d (dP accumulator lane)
  const uint32_t sw = static_cast<uint32_t>(r & 7);

  // fold the dP accumulator of head h and add it to dP_h (one bulk reduce-add)
  auto flush = [&](int h) {
    tc_fence_after();
    float R[Plan::kGWP];
#pragma unroll
    for (int c = 0; c < Plan::kGWP / 32; ++c) {
      uint32_t v[32];
      tmem_ld32(lane_base + Plan::kColsDp + 32 * c, v);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) R[32 * c + i] = __uint_as_float(v[i]);
    }
    if (tid == 0) bulk_wait_group_read<0>();  // the staging tile is no longer read
    __syncthreads();
    if (r < D) {  // row r of dP_h, [d][m] row-major
      const uint32_t row = sbase + Plan::kOut + r * M * 4;
#pragma unroll
      for (int c = 0; c < M / 4; ++c)
        st_shared_v4(row + c * 16, __float_as_uint(R[4 * c] + R[M + 4 * c]),
                     __float_as_uint(R[4 * c + 1] + R[M + 4 * c + 1]),
                     __float_as_uint(R[4 * c + 2] + R[M + 4 * c + 2]),
                     __float_as_uint(R[4 * c + 3] + R[M + 4 * c + 3]));
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      bulk_reduce_add_f32(p.dP + static_cast<size_t>(h) * D * M, sbase + Plan::kOut, D * M * 4);
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
      // rows of [P_h | P_h | 0]: row l holds P_h[l][0 .. m-1] twice, then zeros
      if (r < D) {
        const uint4* src = reinterpret_cast<const uint4*>(p.P + (static_cast<size_t>(x.h) * D + r) * M);
        uint4 pv[M / 8];
#pragma unroll
        for (int c = 0; c < M / 8; ++c) pv[c] = __ldg(src + c);
#pragma unroll
        for (int c = 0; c < Plan::kGWP / 8; ++c) {
          const uint4 w = c < M / 8 ? pv[c] : (c < 2 * M / 8 ? pv[c - M / 8] : make_uint4(0, 0, 0, 0));
          st_shared_v4(sbase + Plan::kP2 + (c / 8) * kFinBox + r * 128 + (((c % 8) ^ sw) << 4), w.x,
                       w.y, w.z, w.w);
        }
      }
      staged_h = x.h;
      dp_fresh = true;
    }
    ok = __syncthreads_and(mbar_wait(&bar_full, i & 1, p.limit_ns));
    if (!ok) break;
    {  // raw fp32 row -> bf16 hi | lo row, in place (everyone reads before anyone writes)
      constexpr int W = Plan::kSlab;
      const uint32_t dsw = dq_slab_swizzle(r, W);
      float v[M];
#pragma unroll
      for (int sl = 0; sl < M / W; ++sl)
#pragma unroll
        for (int q = 0; q < W / 4; ++q) {
          uint32_t t[4];
          ld_shared_v4(sbase + Plan::kG + (sl * kTileRows + r) * W * 4 + ((q ^ dsw) << 4), t);
#pragma unroll
          for (int j = 0; j < 4; ++j) v[sl * W + 4 * q + j] = __uint_as_float(t[j]);
        }
      __syncthreads();
      uint32_t hi[M / 2], lo[M / 2];
#pragma unroll
      for (int j = 0; j < M / 2; ++j) split_pair(v[2 * j], v[2 * j + 1], hi[j], lo[j]);
#pragma unroll
      for (int c = 0; c < Plan::kGWP / 8; ++c) {  // chunk c = values 8c .. 8c + 7 of G's row
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        if (c < M / 8) {
#pragma unroll
          for (int j = 0; j < 4; ++j) w[j] = hi[4 * c + j];
        } else if (c < 2 * M / 8) {
#pragma unroll
          for (int j = 0; j < 4; ++j) w[j] = lo[4 * (c - M / 8) + j];
        }
        st_shared_v4(sbase + Plan::kG + (c / 8) * kFinBox + r * 128 + (((c % 8) ^ sw) << 4), w[0],
                     w[1], w[2], w[3]);
      }
    }
    // the P rows and the converted gradient rows are visible to the tensor
    // cores; the previous unit's reads of tensor memory are done
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      constexpr uint32_t kIdOut = idesc_f16(128, D, kFmtBF16, 0, 0);
      constexpr uint32_t kIdDp = idesc_f16(128, Plan::kGWP, kFmtBF16, 1, 1);
      const uint32_t sG = sbase + Plan::kG, sP = sbase + Plan::kP2, sX = sbase + Plan::kX;
#pragma unroll
      for (int k = 0; k < Plan::kGWP / 16; ++k) {  // out = G [P | P | 0]^T
        const uint32_t off = (k / 4) * kFinBox + (k % 4) * 32;
        mma_ss(tb + Plan::kColsOut, smem_desc(sG + off, 16, 1024, kLayoutSwizzle128),
               smem_desc(sP + off, 16, 1024, kLayoutSwizzle128), kIdOut, k > 0);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k)  // dPacc += X^T G: K = 128 rows in eight steps
        mma_ss(tb + Plan::kColsDp, smem_desc(sX + k * 2048, kFinBox, 1024, kLayoutSwizzle128),
               smem_desc(sG + k * 2048, kFinBox, 1024, kLayoutSwizzle128), kIdDp,
               (dp_fresh && k == 0) ? 0u : 1u);
      // a failure-detection test withholds CTA 0's first "products done":
      // every thread's wait for it runs out, and the CTA takes its abort path
      if (!(p.inject_stall && blockIdx.x == 0 && i == 0)) {
        mma_commit(&bar_mma);
        ++commits;
      }
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
    for (int b = 0; b < D / 32; ++b) {
      uint32_t v[32];
      tmem_ld32(lane_base + Plan::kColsOut + b * 32, v);
      tmem_wait_ld();
      const uint32_t box = sbase + Plan::kOut + (b & 1) * kFinBox;
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
  if (warp == 0) tmem_dealloc(tb, Plan::kCols);
}

template <int D, int M>
cudaError_t launch_fin(const BwdFinishParams& p, cudaStream_t stream) {
  using Plan = FinPlan<D, M>;
  auto kern = bwd_finish_kernel<D, M>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Plan::kLaunch);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0, per_sm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kFinThreads,
                                                         Plan::kLaunch)) != cudaSuccess)
    return e;
  // at most two CTAs per SM: 2 x 256 tensor-memory columns
  per_sm = per_sm < 1 ? 1 : (per_sm > 2 ? 2 : per_sm);
  const long long units = 2LL * p.B * p.H * p.NT;
  const long long cap = static_cast<long long>(per_sm) * sms;
  kern<<<static_cast<unsigned>(units < cap ? units : cap), kFinThreads, Plan::kLaunch, stream>>>(
      p, p.qmap, p.kmap, p.dqmap, p.dkmap);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_fin_d(const BwdFinishParams& p, cudaStream_t stream) {
  switch (p.m) {
    case 16: return launch_fin<D, 16>(p, stream);
    case 32: return launch_fin<D, 32>(p, stream);
    case 64: return launch_fin<D, 64>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool bwd_finish_tc_supported(int d, int m) {
  return (d == 64 || d == 128) && (m == 16 || m == 32 || m == 64);
}

cudaError_t launch_bwd_finish_tc(const BwdFinishParams& p, cudaStream_t stream) {
  if (!bwd_finish_tc_supported(p.d, p.m)) return cudaErrorInvalidValue;
  cudaError_t e = cudaMemsetAsync(p.dP, 0, static_cast<size_t>(p.H) * p.d * p.m * sizeof(float),
                                  stream);
  if (e != cudaSuccess) return e;
  if (2LL * p.B * p.H * p.NT == 0) return cudaSuccess;
  return p.d == 64 ? launch_fin_d<64>(p, stream) : launch_fin_d<128>(p, stream);
}

}  // namespace spa
