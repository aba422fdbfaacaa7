// project.cu -- the projection step  Xp = X P_h  ("Sparse Projection Attention",
// Sec. 3.1.2 and Algorithm 1 steps 2-3; "Projection-Decomposition Attention",
// Algorithm 2.1 step 1).
//
// Two kernels compute it:
//   project_tc_kernel  (bf16 inputs, d a multiple of 8, score-operand output):
//       persistent CTAs, each over a contiguous range of 128-row tiles; X
//       tiles arrive by TMA (128-byte swizzle, K-major) two ahead, P_h^T is
//       written into shared memory in the tensor cores' interleaved layout
//       when the head changes, and one tcgen05 GEMM of shape 128 x m x d per
//       tile accumulates Xp in TMEM (fp32).
//   project_kernel     (any d, fp32 or bf16 inputs, any output mode):
//       SIMT fp32 FMA; thread r of a 128-thread CTA computes row r with P_h
//       staged in shared memory.
// Either way every product of two inputs is exact in fp32 and the sums are
// fp32.  The projection is HBM-bound (about 25 FLOP per byte at d=128, m=32).
//
// Tile modes can also write plain bf16 tiles of Xp (no scale, no multipliers;
// out_b16[which] non-null) in the same pass: the operands of the backward's
// dQp = dS Kp and dKp = dS^T Qp products.
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
//   F16ROWS projected key cache rows (decode): fp16, row-major [BH][rows][m],
//           written at rows pos .. pos+N-1, each row divided by a power of two
//           chosen from its own max |value| (multiplier kept per row).
//   BF16X3  score-GEMM operand tiles in bf16, each value split v = hi + lo
//           (hi = bf16(v), lo = bf16(v - hi)); Q rows are stored [hi|hi|lo] and
//           K rows [hi|lo|hi], so one GEMM of depth 3m sums
//           hi*hi + hi*lo + lo*hi.  Used where fp16 operands are not precise
//           enough (m = 16).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.cuh"
#include "ptx.cuh"
#include "waits.cuh"

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

// Scale, convert and store row `tid` of a score-operand tile, plus its range
// multiplier.  Called by all 128 threads of the CTA (it may synchronise them).
template <int MP, ProjOut MODE, class Sync>
__device__ __forceinline__ void store_tile(const ProjParams& p, float (&acc)[MP], int tile,
                                           int bh, int which, int tid, float* red, Sync sync) {
  constexpr int KD = MODE == ProjOut::BF16X3 ? 3 * MP : MP;
  const int row = tile * kTileRows + tid;
  if constexpr (MODE == ProjOut::F16ROWS) {
    // projected key cache rows: fp16, row-major, one power-of-two multiplier per row
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < MP; ++k) amax = fmaxf(amax, fabsf(acc[k]));
    const int e = range_exponent(amax);
    const float down = pow2i(-e);
    if (row < p.N) {
      const size_t orow = static_cast<size_t>(bh) * p.out_rows + p.out_pos + row;
      uint4* o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out[0]) + orow * MP);
#pragma unroll
      for (int c8 = 0; c8 < MP / 8; ++c8) {
        uint4 w;
        w.x = f16_bits(acc[c8 * 8 + 0] * down) | (static_cast<uint32_t>(f16_bits(acc[c8 * 8 + 1] * down)) << 16);
        w.y = f16_bits(acc[c8 * 8 + 2] * down) | (static_cast<uint32_t>(f16_bits(acc[c8 * 8 + 3] * down)) << 16);
        w.z = f16_bits(acc[c8 * 8 + 4] * down) | (static_cast<uint32_t>(f16_bits(acc[c8 * 8 + 5] * down)) << 16);
        w.w = f16_bits(acc[c8 * 8 + 6] * down) | (static_cast<uint32_t>(f16_bits(acc[c8 * 8 + 7] * down)) << 16);
        o[c8] = w;
      }
      p.mul[0][orow] = pow2i(e);
    }
    return;
  }
  uint16_t* tout = static_cast<uint16_t*>(which == 0 ? p.out[0] : p.out[1]) +
                   (static_cast<size_t>(bh) * p.NT + tile) * (kTileRows * KD);
  if (p.out_b16[which] != nullptr) {  // plain bf16 tile of Xp, same interleaved layout
    uint16_t* bout = static_cast<uint16_t*>(p.out_b16[which]) +
                     (static_cast<size_t>(bh) * p.NT + tile) * (kTileRows * MP);
#pragma unroll
    for (int c8 = 0; c8 < MP / 8; ++c8) {
      uint4 w;
      w.x = bf16_bits(acc[c8 * 8 + 0]) | (static_cast<uint32_t>(bf16_bits(acc[c8 * 8 + 1])) << 16);
      w.y = bf16_bits(acc[c8 * 8 + 2]) | (static_cast<uint32_t>(bf16_bits(acc[c8 * 8 + 3])) << 16);
      w.z = bf16_bits(acc[c8 * 8 + 4]) | (static_cast<uint32_t>(bf16_bits(acc[c8 * 8 + 5])) << 16);
      w.w = bf16_bits(acc[c8 * 8 + 6]) | (static_cast<uint32_t>(bf16_bits(acc[c8 * 8 + 7])) << 16);
      *reinterpret_cast<uint4*>(bout + (c8 * 16 + (tid >> 3)) * 64 + (tid & 7) * 8) = w;
    }
  }
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
      sync();
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

// ------------------------------------------------------------------ SIMT kernel
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
  const T* x = static_cast<const T*>(which == 0 ? p.x[0] : p.x[1]) +
               static_cast<size_t>(bh) * p.N * d;
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

  if constexpr (MODE == ProjOut::F32) {
    const int row = row0 + tid;
    if (row < p.N) {
      float* o = static_cast<float*>(which == 0 ? p.out[0] : p.out[1]) +
                 (static_cast<size_t>(bh) * p.N + row) * m;
#pragma unroll
      for (int k = 0; k < MP; ++k)
        if (k < m) o[k] = acc[k];
    }
  } else {
    store_tile<MP, MODE>(p, acc, tile, bh, which, tid, red, [] { __syncthreads(); });
  }
}

// ------------------------------------------------------------------ tcgen05 kernel
constexpr uint64_t kProjWaitNs = 2000000000ull;

template <int MP, int DCH>
struct ProjTcPlan {
  // X tiles in flight per CTA (three CTAs per SM at m = 32; 3 slots measured
  // C3 37.4 -> 40.6 us, 4 slots 59.8 us: fewer CTAs per SM)
  static constexpr int kSlots = 2;
  static constexpr int kCols = MP < 32 ? 32 : MP;   // TMEM columns (power of 2 >= 32)
  static constexpr int kXBox = kTileRows * 64 * 2;  // one 64-column TMA box: 16 KB
  static constexpr int kXTile = DCH * kXBox;        // one 128-row X tile
  static constexpr int kB = kSlots * kXTile;        // the X tiles in flight, then P_h^T
  static constexpr int kBytes = kB + MP * DCH * 64 * 2 + 1024;
};

// Persistent projection: CTA c takes the contiguous range of units
// [c*U/G, (c+1)*U/G) of the list (tensor, head, 128-row tile), so every CTA
// gets the same number of tiles to within one and re-stages P_h only when
// the head changes.  X tiles (128 rows x d, bf16) arrive by TMA, two ahead,
// into DCH boxes of [128][64] with 128-byte swizzle; B = P_h^T (MP x 64*DCH)
// sits in shared memory in the interleaved K-major layout; one tcgen05 GEMM of
// shape 128 x MP x d per tile accumulates in TMEM, and all 128 threads run
// the epilogue while the next tiles load.
template <int MP, int DCH, ProjOut MODE>
__global__ void __launch_bounds__(128) project_tc_kernel(const ProjParams p,
                                                         const __grid_constant__ CUtensorMap xq,
                                                         const __grid_constant__ CUtensorMap xk) {
  using namespace ptx;
  using Plan = ProjTcPlan<MP, DCH>;
  constexpr int DP = DCH * 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint16_t* sB = reinterpret_cast<uint16_t*>(smem + Plan::kB);  // MP * DP
  constexpr int NS = Plan::kSlots;
  __shared__ uint64_t bar_x[NS], bar_mma;
  __shared__ uint32_t tmem_base_sh;
  __shared__ float red[4];
  const int tid = threadIdx.x, warp = tid >> 5;
  const long long U = static_cast<long long>(p.nx) * p.BH * p.NT;
  const long long G = gridDim.x;
  const long long u0 = blockIdx.x * U / G, u1 = (blockIdx.x + 1) * U / G;
  const uint64_t lim = p.limit_ns ? p.limit_ns : kProjWaitNs;

  // unit -> (tensor, head, tile)
  auto unit_which = [&](long long u) { return static_cast<int>(u / (static_cast<long long>(p.BH) * p.NT)); };
  auto unit_bh = [&](long long u) { return static_cast<int>((u / p.NT) % p.BH); };
  auto unit_tile = [&](long long u) { return static_cast<int>(u % p.NT); };
  int issued = 0, commits = 0;  // thread 0: X copies started, GEMM commits
  auto load = [&](long long u, int slot) {  // thread 0 only
    ++issued;
    const CUtensorMap* xmap = unit_which(u) == 0 ? &xq : &xk;
    uint8_t* dst = smem + slot * Plan::kXTile;
    mbar_arrive_expect_tx(&bar_x[slot], Plan::kXTile);
#pragma unroll
    for (int c = 0; c < DCH; ++c)
      tma_load_3d(dst + c * Plan::kXBox, xmap, c * 64, unit_tile(u) * kTileRows, unit_bh(u),
                  &bar_x[slot]);
  };

  if (warp == 0) {
    tmem_alloc(&tmem_base_sh, Plan::kCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int k = 0; k < NS; ++k) mbar_init(&bar_x[k], 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
    for (int k = 0; k < NS; ++k)
      if (u0 + k < u1) load(u0 + k, k);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tmem_base_sh;

  bool ok = true;
  int staged_h = -1;
  for (long long u = u0; ok && u < u1; ++u) {
    const int i = static_cast<int>(u - u0), slot = i % NS;
    const int which = unit_which(u), bh = unit_bh(u), tile = unit_tile(u);
    const int h = bh % p.H;
    if (h != staged_h) {
      // B operand: element (n, k) = P_h[k][n] at ((k/8)*(MP/8) + n/8)*64 + (n%8)*8 + k%8.
      // The previous GEMM has completed (waited below), so sB is free.  Each
      // thread reads 8 consecutive n of one row k of P_h (16 bytes; m == MP is
      // a multiple of 8 and P is 16-byte aligned) and all its reads are issued
      // before the first store, so the L2 latency is paid about once.
      const uint4* P = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.P) +
                                                      static_cast<size_t>(h) * p.d * MP);
      constexpr int kVec = MP * DP / 8;  // 16-byte pieces of P_h^T (zero rows past d)
      constexpr int kPer = (kVec + 127) / 128;
      uint4 pv[kPer];
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int e = tid + i * 128, k = e / (MP / 8), n0 = (e % (MP / 8)) * 8;
        pv[i] = (e < kVec && k < p.d) ? __ldg(P + (static_cast<size_t>(k) * MP + n0) / 8)
                                      : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int e = tid + i * 128, k = e / (MP / 8), n0 = (e % (MP / 8)) * 8;
        if (e < kVec) {
          uint16_t* dst = sB + ((k >> 3) * (MP / 8) + (n0 >> 3)) * 64 + (k & 7);
          const uint32_t w[4] = {pv[i].x, pv[i].y, pv[i].z, pv[i].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            dst[(2 * q) * 8] = static_cast<uint16_t>(w[q] & 0xFFFFu);
            dst[(2 * q + 1) * 8] = static_cast<uint16_t>(w[q] >> 16);
          }
        }
      }
      fence_proxy_async_smem();
      __syncthreads();
      staged_h = h;
    }
    ok = __syncthreads_and(mbar_wait(&bar_x[slot], (i / NS) & 1, lim));
    if (!ok) break;
    if (tid == 0) {
      constexpr uint32_t idesc = idesc_f16(128, MP, kFmtBF16, 0, 0);
      const uint32_t sx = smem_u32(smem + slot * Plan::kXTile);
      tc_fence_after();
#pragma unroll
      for (int st = 0; st < DP / 16; ++st) {
        const uint64_t ad = smem_desc(sx + (st >> 2) * Plan::kXBox + (st & 3) * 32, 16, 1024,
                                      kLayoutSwizzle128);
        const uint64_t bd = smem_desc(smem_u32(sB) + st * 2 * (MP / 8) * 128, (MP / 8) * 128, 128,
                                      kLayoutInterleave);
        mma_ss(tb, ad, bd, idesc, st > 0);
      }
      // a failure-detection test withholds CTA 0's first "GEMM done": every
      // thread's wait for it runs out, and the CTA takes its abort path
      if (!(p.inject_stall && blockIdx.x == 0 && i == 0)) {
        mma_commit(&bar_mma);
        ++commits;
      }
    }
    ok = __syncthreads_and(mbar_wait(&bar_mma, i & 1, lim));
    if (!ok) break;
    // the GEMM has read X slot `slot`: refill it NS tiles ahead
    if (tid == 0 && u + NS < u1) load(u + NS, slot);
    tc_fence_after();
    float acc[MP];
#pragma unroll
    for (int c = 0; c < MP; c += 16) {
      uint32_t r[16];
      tmem_ld16(tb + (static_cast<uint32_t>(warp * 32) << 16) + c, r);
      tmem_wait_ld();
#pragma unroll
      for (int q = 0; q < 16; ++q) acc[c + q] = __uint_as_float(r[q]);
    }
    // every thread's accumulator is read before the next GEMM overwrites it
    tc_fence_before();
    __syncthreads();
    store_tile<MP, MODE>(p, acc, tile, bh, which, tid, red, [] { __syncthreads(); });
  }
  if (tid == 0 && !ok) {
    atomicExch(p.err, 1);
    // a GEMM may still be in flight: let it finish before TMEM is released
    mma_commit(&bar_mma);
    mbar_wait(&bar_mma, commits & 1, lim);
  }
  // every X copy started lands before the CTA's memory is released (all of
  // them already have unless a wait gave up): the last copy into each slot
  if (tid == 0)
    for (int i = max(0, issued - NS); i < issued; ++i)
      mbar_wait(&bar_x[i % NS], (i / NS) & 1, lim);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, Plan::kCols);
}

// ------------------------------------------------------------------ warp-specialised tcgen05 kernel
// One CTA per SM over a contiguous range of units (tensor, head, 128-row
// tile), with the roles apart so that the copies never wait for the
// epilogue:
//   warps 0-7  two epilogue warpgroups, tile i to warpgroup i % 2: the tile's
//              accumulator out of TMEM (one row per thread), then the range
//              exponent, conversion and stores of store_tile
//   warp  8    loads (one thread): X tiles by TMA into a ring of kSlots
//   warp  9    TMEM allocation; one thread issues each tile's 128 x MP x d
//              GEMM into one of four TMEM accumulators (two per epilogue
//              warpgroup)
// The loader starts at once; the other warps write P_h^T of every head the
// range touches (at most kWsHeads) into shared memory and meet before the
// first GEMM.  Used where m != 32: at m = 64 it measured 158 -> 131 us on
// C4's projection, at m = 128 251 -> 206 us (C5), at m = 16 126 -> 118 us; at
// m = 32, where the per-CTA kernel runs three CTAs per SM, it was slower
// (C3 33.4 -> 37 us) and the per-CTA kernel is kept.
constexpr int kWsHeads = 3;
constexpr int kWsEpi = 2;  // epilogue warpgroups: tile i goes to warpgroup i % kWsEpi
constexpr int kWsThreads = 128 * kWsEpi + 64;
template <int MP, int DCH>
struct ProjWsPlan {
  static constexpr int kCols = MP < 32 ? 32 : MP;   // one accumulator's TMEM columns
  static constexpr int kAcc = 2 * kWsEpi;           // accumulators: two per epilogue warpgroup
  static constexpr int kTmem = kAcc * kCols <= 32 ? 32 : kAcc * kCols <= 64 ? 64 : kAcc * kCols <= 128 ? 128 : kAcc * kCols <= 256 ? 256 : 512;
  static constexpr int kXBox = kTileRows * 64 * 2;  // one 64-column TMA box: 16 KB
  static constexpr int kXTile = DCH * kXBox;
  static constexpr int kPT = MP * DCH * 64 * 2;     // one head's P_h^T
  static constexpr int kMax = 227 * 1024 - 2048;
  static constexpr int kSlotsFit = (kMax - kWsHeads * kPT) / kXTile;
  static constexpr bool kOk = kSlotsFit >= 2 && kAcc * kCols <= 512;  // else the per-CTA kernel
  static constexpr int kSlots = kSlotsFit > 6 ? 6 : kSlotsFit < 2 ? 2 : kSlotsFit;
  static constexpr int kB = kSlots * kXTile;
  static constexpr int kBytes = kB + kWsHeads * kPT + 1024;
};

template <int MP, int DCH, ProjOut MODE>
__global__ void __launch_bounds__(kWsThreads, 1) project_ws_kernel(const ProjParams p,
                                                            const __grid_constant__ CUtensorMap xq,
                                                            const __grid_constant__ CUtensorMap xk) {
  using namespace ptx;
  using Plan = ProjWsPlan<MP, DCH>;
  constexpr int DP = DCH * 64;
  constexpr int NS = Plan::kSlots;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  constexpr int NA = Plan::kAcc;
  constexpr int kLoadW = 4 * kWsEpi, kMmaW = kLoadW + 1;
  __shared__ uint64_t x_full[NS], x_empty[NS], acc_full[NA], acc_empty[NA], drain;
  __shared__ uint32_t tmem_base_sh;
  __shared__ float red[kWsEpi][2][4];
  __shared__ volatile int abort_sh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long U = static_cast<long long>(p.nx) * p.BH * p.NT;
  const long long G = gridDim.x;
  const long long u0 = blockIdx.x * U / G, u1 = (blockIdx.x + 1) * U / G;
  auto unit_which = [&](long long u) {
    return static_cast<int>(u / (static_cast<long long>(p.BH) * p.NT));
  };
  auto unit_bh = [&](long long u) { return static_cast<int>((u / p.NT) % p.BH); };
  auto unit_tile = [&](long long u) { return static_cast<int>(u % p.NT); };
  // heads of the range in order of first use; a unit's P_h^T buffer is the
  // index of its head in that list
  const int h_first = unit_bh(u0) % p.H;
  const WaitCtl ctl{&abort_sh, p.err, p.limit_ns ? p.limit_ns : kProjWaitNs};

  if (warp == kMmaW) {
    tmem_alloc(&tmem_base_sh, Plan::kTmem);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int k = 0; k < NS; ++k) {
      mbar_init(&x_full[k], 1);
      mbar_init(&x_empty[k], 1);
    }
    for (int k = 0; k < NA; ++k) {
      mbar_init(&acc_full[k], 1);
      mbar_init(&acc_empty[k], 4);  // one arrival per warp of the epilogue warpgroup
    }
    mbar_init(&drain, 1);
    abort_sh = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tmem_base_sh;
  // The loader starts at once; the other warps write P_h^T of every head of
  // the range meanwhile and meet at a named barrier before the first GEMM.
  if (warp != kLoadW) {
  // P_h^T of every head of the range: element (n, k) = P_h[k][n] at
  // ((k/8)*(MP/8) + n/8)*64 + (n%8)*8 + k%8, rows past d zero
  if (u0 < u1) {
    int hs[kWsHeads];
    int nh = 0, hprev = -1;
    for (long long v = u0; v < u1 && nh <= kWsHeads; v = (v / p.NT + 1) * p.NT) {
      const int h = unit_bh(v) % p.H;
      if (h != hprev) {
        if (nh < kWsHeads) hs[nh] = h;
        ++nh;
        hprev = h;
      }
    }
    constexpr int kVec = MP * DP / 8;  // 16-byte pieces of one P_h^T
    for (int hh = 0; hh < nh && hh < kWsHeads; ++hh) {
      const uint4* P = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.P) +
                                                      static_cast<size_t>(hs[hh]) * p.d * MP);
      uint16_t* sB = reinterpret_cast<uint16_t*>(smem + Plan::kB + hh * Plan::kPT);
      // builder index: every thread but the loader warp's
      for (int e = warp < kLoadW ? tid : tid - 32; e < kVec; e += kWsThreads - 32) {
        const int k = e / (MP / 8), n0 = (e % (MP / 8)) * 8;
        const uint4 pv = k < p.d ? __ldg(P + (static_cast<size_t>(k) * MP + n0) / 8)
                                 : make_uint4(0u, 0u, 0u, 0u);
        uint16_t* dst = sB + ((k >> 3) * (MP / 8) + (n0 >> 3)) * 64 + (k & 7);
        const uint32_t w[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          dst[(2 * q) * 8] = static_cast<uint16_t>(w[q] & 0xFFFFu);
          dst[(2 * q + 1) * 8] = static_cast<uint16_t>(w[q] >> 16);
        }
      }
    }
    fence_proxy_async_smem();
  }
    named_bar_sync(15, kWsThreads - 32);
    tc_fence_after();
  }

  if (warp == kLoadW) {
    // ---------------------------------------------------------------- loads
    if (lane == 0) {
      long long issued = 0;
      for (long long u = u0; u < u1; ++u) {
        const int i = static_cast<int>(u - u0), slot = i % NS;
        if (i >= NS && !wait_or_abort(&x_empty[slot], ((i / NS) - 1) & 1, ctl)) break;
        ++issued;
        const CUtensorMap* xmap = unit_which(u) == 0 ? &xq : &xk;
        uint8_t* dst = smem + slot * Plan::kXTile;
        mbar_arrive_expect_tx(&x_full[slot], Plan::kXTile);
#pragma unroll
        for (int c = 0; c < DCH; ++c)
          tma_load_3d(dst + c * Plan::kXBox, xmap, c * 64, unit_tile(u) * kTileRows, unit_bh(u),
                      &x_full[slot]);
      }
      // every copy started lands before the CTA's memory is released
      for (long long i = issued > NS ? issued - NS : 0; i < issued; ++i)
        mbar_wait(&x_full[i % NS], (i / NS) & 1, ctl.limit_ns);
    }
  } else if (warp == kMmaW) {
    // ---------------------------------------------------------------- MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16(128, MP, kFmtBF16, 0, 0);
      int hslot = 0, hprev = h_first;
      for (long long u = u0; u < u1; ++u) {
        const int i = static_cast<int>(u - u0), slot = i % NS, ab = i % NA;
        const int h = unit_bh(u) % p.H;
        if (h != hprev) { ++hslot; hprev = h; }
        if (!wait_or_abort(&x_full[slot], (i / NS) & 1, ctl)) break;
        if (i >= NA && !wait_or_abort(&acc_empty[ab], ((i / NA) - 1) & 1, ctl)) break;
        tc_fence_after();
        const uint32_t sx = smem_u32(smem + slot * Plan::kXTile);
        const uint32_t sb = smem_u32(smem + Plan::kB + hslot * Plan::kPT);
#pragma unroll
        for (int st = 0; st < DP / 16; ++st) {
          const uint64_t ad = smem_desc(sx + (st >> 2) * Plan::kXBox + (st & 3) * 32, 16, 1024,
                                        kLayoutSwizzle128);
          const uint64_t bd = smem_desc(sb + st * 2 * (MP / 8) * 128, (MP / 8) * 128, 128,
                                        kLayoutInterleave);
          mma_ss(tb + ab * Plan::kCols, ad, bd, idesc, st > 0);
        }
        mma_commit(&x_empty[slot]);  // the X tile is read
        // a failure-detection test withholds CTA 0's first "accumulator
        // ready": its epilogue warpgroup gives up, and every role aborts
        if (!(p.inject_stall && blockIdx.x == 0 && i == 0)) mma_commit(&acc_full[ab]);
      }
      mma_commit(&drain);
      mbar_wait(&drain, 0, ctl.limit_ns);  // own MMAs in flight
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int eg = warp >> 2;  // this epilogue warpgroup takes units eg, eg + kWsEpi, ...
    const int et = tid & 127;
    for (long long u = u0 + eg; u < u1; u += kWsEpi) {
      const int i = static_cast<int>(u - u0), ab = i % NA;
      // the warpgroup decides together, so that its four warps meet the
      // named barrier of store_tile as one (a thread that gave up has set abort_sh)
      const uint32_t bar = 1 + eg;
      __syncwarp();
      if (!named_bar_and(bar, 128, wait_or_abort(&acc_full[ab], (i / NA) & 1, ctl))) break;
      tc_fence_after();
      float acc[MP];
#pragma unroll
      for (int c = 0; c < MP; c += 16) {
        uint32_t r[16];
        tmem_ld16(tb + ab * Plan::kCols + (static_cast<uint32_t>((warp & 3) * 32) << 16) + c, r);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 16; ++q) acc[c + q] = __uint_as_float(r[q]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[ab]);  // the accumulator may take unit i+2
      store_tile<MP, MODE>(p, acc, unit_tile(u), unit_bh(u), unit_which(u), et,
                           red[eg][(i / kWsEpi) & 1], [bar] { named_bar_sync(bar, 128); });
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaW) tmem_dealloc(tb, Plan::kTmem);
}

template <int MP, int DCH, ProjOut MODE>
cudaError_t launch_ws_one(const ProjParams& p, cudaStream_t stream) {
  using Plan = ProjWsPlan<MP, DCH>;
  auto kern = project_ws_kernel<MP, DCH, MODE>;
  const int smem = Plan::kBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  const long long units = static_cast<long long>(p.nx) * p.BH * p.NT;
  const long long grid = units < sms ? units : sms;
  if (grid <= 0) return cudaSuccess;
  kern<<<static_cast<unsigned>(grid), kWsThreads, smem, stream>>>(p, p.xmap[0], p.xmap[1]);
  return cudaGetLastError();
}

// Whether every CTA's range of units touches at most kWsHeads heads.
bool project_ws_fits(const ProjParams& p, int sms) {
  const long long units = static_cast<long long>(p.nx) * p.BH * p.NT;
  if (units <= 0 || sms <= 0) return false;
  const long long G = units < sms ? units : sms;
  const long long per = (units + G - 1) / G;
  return per / p.NT + 2 <= kWsHeads;
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

template <int MP, int DCH, ProjOut MODE>
cudaError_t launch_tc_one(const ProjParams& p, cudaStream_t stream) {
  using Plan = ProjTcPlan<MP, DCH>;
  auto kern = project_tc_kernel<MP, DCH, MODE>;
  const int smem = Plan::kBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // the whole unified L1 as shared memory, so that several CTAs are resident
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0, per_sm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 128, smem)) != cudaSuccess)
    return e;
  // The occupancy query may assume the default L1 / shared split; with the
  // whole carveout as shared memory, this many CTAs fit by shared memory.
  int sm_smem = 0, reserved = 0;
  if ((e = cudaDeviceGetAttribute(&sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) !=
          cudaSuccess ||
      (e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev)) !=
          cudaSuccess)
    return e;
  per_sm = max(per_sm, sm_smem / (smem + reserved));
  // never more CTAs per SM than their TMEM allocations fit in 512 columns
  per_sm = max(1, min(per_sm, 512 / Plan::kCols));
  const long long units = static_cast<long long>(p.nx) * p.BH * p.NT;
  const long long grid = min(units, static_cast<long long>(sms) * per_sm);
  if (grid <= 0) return cudaSuccess;
  kern<<<static_cast<unsigned>(grid), 128, smem, stream>>>(p, p.xmap[0], p.xmap[1]);
  return cudaGetLastError();
}

template <int MP, ProjOut MODE>
cudaError_t launch_tc_mp(const ProjParams& p, cudaStream_t stream) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
      MP != 32 && project_ws_fits(p, sms)) {
    switch ((p.d + 63) / 64) {
      case 1: if constexpr (ProjWsPlan<MP, 1>::kOk) return launch_ws_one<MP, 1, MODE>(p, stream); break;
      case 2: if constexpr (ProjWsPlan<MP, 2>::kOk) return launch_ws_one<MP, 2, MODE>(p, stream); break;
      case 3: if constexpr (ProjWsPlan<MP, 3>::kOk) return launch_ws_one<MP, 3, MODE>(p, stream); break;
      case 4: if constexpr (ProjWsPlan<MP, 4>::kOk) return launch_ws_one<MP, 4, MODE>(p, stream); break;
      default: return cudaErrorInvalidValue;
    }
  }
  switch ((p.d + 63) / 64) {
    case 1: return launch_tc_one<MP, 1, MODE>(p, stream);
    case 2: return launch_tc_one<MP, 2, MODE>(p, stream);
    case 3: return launch_tc_one<MP, 3, MODE>(p, stream);
    case 4: return launch_tc_one<MP, 4, MODE>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
cudaError_t launch_f32_out(const ProjParams& p, cudaStream_t stream) {
  if (p.m <= 16) return launch_one<T, 16, ProjOut::F32>(p, stream);
  if (p.m <= 32) return launch_one<T, 32, ProjOut::F32>(p, stream);
  if (p.m <= 64) return launch_one<T, 64, ProjOut::F32>(p, stream);
  return launch_one<T, 128, ProjOut::F32>(p, stream);
}

}  // namespace

bool project_tc_eligible(const ProjParams& p) {
  return p.bf16_in && p.mode != ProjOut::F32 && p.d % 8 == 0 && p.d <= 256;
}

cudaError_t launch_project(const ProjParams& p, cudaStream_t stream) {
  if (p.mode == ProjOut::F32)
    return p.bf16_in ? launch_f32_out<__nv_bfloat16>(p, stream) : launch_f32_out<float>(p, stream);
  if (!p.bf16_in) return cudaErrorInvalidValue;
  const bool tc = p.use_tc && project_tc_eligible(p);
  if (p.mode == ProjOut::F16ROWS) {
    switch (p.m) {
      case 16:
        return tc ? launch_tc_mp<16, ProjOut::F16ROWS>(p, stream)
                  : launch_one<__nv_bfloat16, 16, ProjOut::F16ROWS>(p, stream);
      case 32:
        return tc ? launch_tc_mp<32, ProjOut::F16ROWS>(p, stream)
                  : launch_one<__nv_bfloat16, 32, ProjOut::F16ROWS>(p, stream);
      case 64:
        return tc ? launch_tc_mp<64, ProjOut::F16ROWS>(p, stream)
                  : launch_one<__nv_bfloat16, 64, ProjOut::F16ROWS>(p, stream);
      case 128:
        return tc ? launch_tc_mp<128, ProjOut::F16ROWS>(p, stream)
                  : launch_one<__nv_bfloat16, 128, ProjOut::F16ROWS>(p, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  if (p.mode == ProjOut::BF16X3) {
    if (p.m != 16) return cudaErrorInvalidValue;
    return tc ? launch_tc_mp<16, ProjOut::BF16X3>(p, stream)
              : launch_one<__nv_bfloat16, 16, ProjOut::BF16X3>(p, stream);
  }
  switch (p.m) {
    case 32:
      return tc ? launch_tc_mp<32, ProjOut::F16X1>(p, stream)
                : launch_one<__nv_bfloat16, 32, ProjOut::F16X1>(p, stream);
    case 64:
      return tc ? launch_tc_mp<64, ProjOut::F16X1>(p, stream)
                : launch_one<__nv_bfloat16, 64, ProjOut::F16X1>(p, stream);
    case 128:
      return tc ? launch_tc_mp<128, ProjOut::F16X1>(p, stream)
                : launch_one<__nv_bfloat16, 128, ProjOut::F16X1>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace spa
