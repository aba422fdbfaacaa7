// topk.cu -- row-wise Top-k feature sparsification (Sparse Feature Attention
// notes, Sec. 1 "feature sparsification": every query / key row keeps its k
// coordinates of largest magnitude and zeroes the rest; attention then runs
// on the sparsified rows at scale 1/sqrt(d)).
//
// bf16 rows of up to 128 features take a thread per row and a search on bit
// planes (below); other rows a
// warp per row of d = 32 * E features, lane l holding the E consecutive
// features E*l .. E*l + E - 1.  The k-th largest magnitude T is found by a
// binary search over the magnitude's bit pattern (for non-negative floats the
// bit pattern orders like the value).  Every
// feature with |x| > T is kept, and of the features with |x| == T the ones
// with the lowest indices, as many as k still needs (a warp-wide exclusive
// scan in index order).  The selection is made on the exact input values, so
// it is bit-exact and deterministic.
#include <cuda_bf16.h>
#include <stdint.h>

#include "kernels.cuh"
#include "ptx.cuh"

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

// Delta swap: exchange the bits of x selected by m with those s places above.
__device__ __forceinline__ uint32_t delta_swap(uint32_t x, int s, uint32_t m) {
  const uint32_t t = (x ^ (x >> s)) & m;
  return x ^ t ^ (t << s);
}
// Bit b = 16h + w of a group mask stands for feature 2w + h of the group (the
// order the bit-plane transpose leaves); `to_index_order` interleaves the two
// halves (bit 16h + w -> bit 2w + h), `to_plane_order` undoes it.
__device__ __forceinline__ uint32_t to_index_order(uint32_t x) {
  x = delta_swap(x, 8, 0x0000FF00u);
  x = delta_swap(x, 4, 0x00F000F0u);
  x = delta_swap(x, 2, 0x0C0C0C0Cu);
  return delta_swap(x, 1, 0x22222222u);
}
__device__ __forceinline__ uint32_t to_plane_order(uint32_t x) {
  x = delta_swap(x, 1, 0x22222222u);
  x = delta_swap(x, 2, 0x0C0C0C0Cu);
  x = delta_swap(x, 4, 0x00F000F0u);
  return delta_swap(x, 8, 0x0000FF00u);
}
// In-place transpose of the two 16 x 16 bit matrices held in the halves of
// x[0..15] (row = word, column = bit within the half): afterwards bit c of
// half h of x[r] is the former bit r of half h of x[c].
__device__ __forceinline__ void transpose16x2(uint32_t (&x)[16]) {
#pragma unroll
  for (int level = 0; level < 4; ++level) {
    const int s = 8 >> level;
    const uint32_t m = level == 0 ? 0x00FF00FFu : level == 1 ? 0x0F0F0F0Fu
                     : level == 2 ? 0x33333333u : 0x55555555u;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i & s) continue;
      const uint32_t t = ((x[i] >> s) ^ x[i + s]) & m;
      x[i + s] ^= t;
      x[i] ^= t << s;
    }
  }
}

// Top-k of one bf16 row of 32 G features held by one thread, as G groups of
// 32 features (16 words of two; sign bits may be set).  The magnitudes of a
// group are transposed into bit planes: word b of a group becomes the mask of
// its features whose magnitude has bit b set.  The threshold search of the
// warp kernel then runs on masks: E holds the features whose magnitude agrees
// with the threshold t above the current bit, Gm the ones already known to be
// larger; count(|x| >= t | 2^b) = |Gm| + popc(E & plane_b).  Each of the 15
// steps costs a few instructions per 32 features instead of one or more per
// feature.  Ties at t (E at the end) are kept lowest index first, as many as
// k - |Gm| needs, as in the warp kernel, so both give the same bits.  On
// return keep[g] has bits w and 16 + w set for the kept features 2w and
// 2w + 1 of group g.
template <int G>
__device__ __forceinline__ void select_row(uint32_t (&a)[G][16], int k, uint32_t (&keep)[G]) {
#pragma unroll
  for (int g = 0; g < G; ++g) {
#pragma unroll
    for (int w = 0; w < 16; ++w) a[g][w] &= 0x7fff7fffu;
    transpose16x2(a[g]);
  }
  // largest t with count(|x| >= t) >= k, bit by bit from the top, on the planes
  uint32_t E[G], Gm[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    E[g] = 0xffffffffu;
    Gm[g] = 0u;
  }
  int greater = 0;  // popc of Gm
#pragma unroll
  for (int b = 14; b >= 0; --b) {
    uint32_t Eb[G];
    int c = greater;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      Eb[g] = E[g] & a[g][b];
      c += __popc(Eb[g]);
    }
    const bool set = c >= k;  // bit b of t is 1
#pragma unroll
    for (int g = 0; g < G; ++g) {
      Gm[g] = set ? Gm[g] : (Gm[g] | Eb[g]);
      E[g] = set ? Eb[g] : (E[g] & ~a[g][b]);
    }
    greater = set ? greater : c;
  }
  // the ties, lowest feature index first, as many as k still needs
  int need = k - greater;  // >= 1: fewer than k magnitudes exceed t
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const uint32_t eo = to_index_order(E[g]);
    const int pc = __popc(eo);
    uint32_t sel = 0u;
    if (need >= pc) {
      sel = eo;
      need -= pc;
    } else if (need > 0) {
      uint32_t rest = eo;
      for (int i = 0; i < need; ++i) rest &= rest - 1u;  // drop the lowest `need`
      sel = eo & ~rest;
      need = 0;
    }
    keep[g] = Gm[g] | to_plane_order(sel);
  }
}
// Word w of group g (features 2w, 2w + 1) with the dropped halves zeroed.
template <int G>
__device__ __forceinline__ uint32_t kept_word(uint32_t v, const uint32_t (&keep)[G], int g, int w) {
  return v & (((keep[g] >> w) & 0x00010001u) * 0xFFFFu);
}

// bf16 rows of 32 features: one thread per row, straight from global memory
// (a row is 64 bytes, so the 16-byte loads of a warp are half coalesced).
__global__ void __launch_bounds__(128) topk_rows32_bf16_kernel(const uint16_t* __restrict__ x,
                                                               uint16_t* __restrict__ y,
                                                               long long rows, int k) {
  const long long row = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (row >= rows) return;
  const uint4* src = reinterpret_cast<const uint4*>(x + row * 32);
  uint32_t a[1][16];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 u = __ldg(src + i);
    a[0][4 * i] = u.x;
    a[0][4 * i + 1] = u.y;
    a[0][4 * i + 2] = u.z;
    a[0][4 * i + 3] = u.w;
  }
  uint32_t keep[1];
  select_row<1>(a, k, keep);
  uint4* dst = reinterpret_cast<uint4*>(y + row * 32);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 u = __ldg(src + i);
    dst[i] = make_uint4(kept_word<1>(u.x, keep, 0, 4 * i), kept_word<1>(u.y, keep, 0, 4 * i + 1),
                        kept_word<1>(u.z, keep, 0, 4 * i + 2),
                        kept_word<1>(u.w, keep, 0, 4 * i + 3));
  }
}

// bf16 rows of 64 or 128 features: one thread per row, a block's 128 rows
// (contiguous in memory) passing through shared memory with 16-byte accesses
// that are coalesced across the block.  In shared memory 16-byte chunk c of
// row r sits at chunk c ^ (r % 8), so that the eight threads of a quarter
// warp (eight consecutive rows, same chunk) and eight consecutive chunks of
// the coalesced passes both fall in eight different bank groups.
template <int D>
__global__ void __launch_bounds__(128) topk_rows_bf16_kernel(const uint16_t* __restrict__ x,
                                                             uint16_t* __restrict__ y,
                                                             long long rows, int k) {
  constexpr int G = D / 32, V = D / 8;  // groups of 32 features, 16-byte chunks of a row
  static_assert(V >= 8, "eight-chunk swizzle");
  __shared__ uint4 tile[128 * V];
  const int tid = threadIdx.x;
  const long long row0 = static_cast<long long>(blockIdx.x) * 128;
  const int nrows = static_cast<int>(min(128LL, rows - row0));
  auto slot = [](int r, int c) { return r * V + (c ^ (r & 7)); };
  const uint4* src = reinterpret_cast<const uint4*>(x + row0 * D);
  for (int q = tid; q < nrows * V; q += 128) tile[slot(q / V, q % V)] = __ldg(src + q);
  __syncthreads();
  if (tid < nrows) {
    uint32_t a[G][16];
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const uint4 u = tile[slot(tid, i)];
      const int g = i / 4, w = (i % 4) * 4;  // four chunks per group
      a[g][w] = u.x;
      a[g][w + 1] = u.y;
      a[g][w + 2] = u.z;
      a[g][w + 3] = u.w;
    }
    uint32_t keep[G];
    select_row<G>(a, k, keep);
    // read the row again rather than keep it in registers through the search
    asm volatile("" ::: "memory");
#pragma unroll
    for (int i = 0; i < V; ++i) {  // each thread rewrites only its own row's slots
      const uint4 u = tile[slot(tid, i)];
      const int g = i / 4, w = (i % 4) * 4;
      tile[slot(tid, i)] = make_uint4(kept_word<G>(u.x, keep, g, w), kept_word<G>(u.y, keep, g, w + 1),
                                      kept_word<G>(u.z, keep, g, w + 2),
                                      kept_word<G>(u.w, keep, g, w + 3));
    }
  }
  __syncthreads();
  uint4* dst = reinterpret_cast<uint4*>(y + row0 * D);
  for (int q = tid; q < nrows * V; q += 128) dst[q] = tile[slot(q / V, q % V)];
}

// bf16 rows of 64 or 128 features, persistent: a CTA walks blocks of 128 rows
// (blockIdx.x, + gridDim.x, ...) through two shared-memory buffers.  One
// thread brings a block in by TMA (64-feature boxes, 128-byte swizzle: chunk
// c of row r at chunk c ^ (r % 8) of its box row, so the per-row reads of a
// quarter warp hit eight bank groups) two blocks ahead; every thread selects
// its row (select_row) and writes the kept values back over the same slots;
// the block leaves by TMA stores (rows past the end are clipped), and the
// buffer is refilled once those stores have read it.  Bounded waits: a wait
// that runs out sets the device error word, and the CTA lets its own copies
// land before it exits.
template <int D>
__global__ void __launch_bounds__(128) topk_rows_bf16_tma_kernel(
    const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap ymap,
    long long nblocks, int k, int* err, unsigned long long limit_ns, int inject_stall) {
  using namespace ptx;
  constexpr int G = D / 32, V = D / 8, NB = D / 64;  // groups, 16-byte chunks, boxes per row
  constexpr int kBox = 128 * 128;                    // one box: 128 rows x 128 bytes
  constexpr int kBuf = NB * kBox;                    // one block of 128 rows
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[2];
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* sptr = smem_raw + (sbase - smem_u32(smem_raw));
  const int tid = threadIdx.x;
  const long long step = gridDim.x;
  int issued0 = 0, issued1 = 0;  // thread 0: loads started into buffer 0 / 1
  auto load = [&](long long blk, int s) {
    mbar_arrive_expect_tx(&full[s], kBuf);
    // a failure-detection test arms CTA 0's first buffer without starting its
    // copies: the wait for it runs out, and nothing is left in flight
    if (!(inject_stall && blockIdx.x == 0 && s == 0 && issued0 == 0)) {
#pragma unroll
      for (int h = 0; h < NB; ++h)
        tma_load_3d(sptr + s * kBuf + h * kBox, &xmap, h * 64, static_cast<int>(blk * 128), 0,
                    &full[s]);
    }
    if (s == 0) ++issued0;
    else ++issued1;
  };
  if (tid == 0) {
    prefetch_tmap(&xmap);
    prefetch_tmap(&ymap);
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    fence_mbar_init();
  }
  __syncthreads();
  const long long b0 = blockIdx.x;
  if (tid == 0) {
    if (b0 < nblocks) load(b0, 0);
    if (b0 + step < nblocks) load(b0 + step, 1);
  }
  const uint32_t sw = static_cast<uint32_t>(tid & 7);
  bool ok = true;
  int i = 0;
  for (long long b = b0; b < nblocks; b += step, ++i) {
    const int s = i & 1;
    ok = __syncthreads_and(mbar_wait(&full[s], (i >> 1) & 1, limit_ns));
    if (!ok) break;
    const uint32_t row = sbase + s * kBuf + tid * 128;  // this thread's row in box 0
    uint32_t a[G][16];
#pragma unroll
    for (int c = 0; c < V; ++c) {
      uint32_t t[4];
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(t[0]), "=r"(t[1]), "=r"(t[2]), "=r"(t[3])
                   : "r"(row + (c / 8) * kBox + (((c % 8) ^ sw) << 4)));
#pragma unroll
      for (int e = 0; e < 4; ++e) a[c / 4][(c % 4) * 4 + e] = t[e];
    }
    uint32_t keep[G];
    select_row<G>(a, k, keep);
    // read the row again rather than keep it in registers through the search
    asm volatile("" ::: "memory");
#pragma unroll
    for (int c = 0; c < V; ++c) {
      const uint32_t addr = row + (c / 8) * kBox + (((c % 8) ^ sw) << 4);
      uint32_t t[4];
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(t[0]), "=r"(t[1]), "=r"(t[2]), "=r"(t[3])
                   : "r"(addr));
      const int g = c / 4, w = (c % 4) * 4;
      st_shared_v4(addr, kept_word<G>(t[0], keep, g, w), kept_word<G>(t[1], keep, g, w + 1),
                   kept_word<G>(t[2], keep, g, w + 2), kept_word<G>(t[3], keep, g, w + 3));
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
#pragma unroll
      for (int h = 0; h < NB; ++h)
        tma_store_3d(&ymap, sbase + s * kBuf + h * kBox, h * 64, static_cast<int>(b * 128), 0);
      bulk_commit_group();
      if (b + 2 * step < nblocks) {
        bulk_wait_group_read<0>();  // the stores have read this buffer
        load(b + 2 * step, s);
      }
    }
  }
  if (tid == 0) {
    if (!ok) atomicExch(err, 1);
    // loads started and not consumed land before the CTA's memory is released
    // (i iterations ran to completion: (i + 1) / 2 of them used buffer 0, i / 2 buffer 1)
    if (issued0 > (i + 1) / 2) mbar_wait(&full[0], (issued0 - 1) & 1, limit_ns);
    if (issued1 > i / 2) mbar_wait(&full[1], (issued1 - 1) & 1, limit_ns);
    bulk_wait_group_read<0>();
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

template <int D>
cudaError_t launch_bf16_rows_staged(const TopkParams& p, cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>((p.rows + 127) / 128);
  const uint16_t* x = static_cast<const uint16_t*>(p.x);
  uint16_t* y = static_cast<uint16_t*>(p.y);
  if constexpr (D == 32)
    topk_rows32_bf16_kernel<<<grid, 128, 0, stream>>>(x, y, p.rows, p.k);
  else
    topk_rows_bf16_kernel<D><<<grid, 128, 0, stream>>>(x, y, p.rows, p.k);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_bf16_rows_tma(const TopkParams& p, cudaStream_t stream) {
  constexpr int kSmem = 2 * (D / 64) * 128 * 128 + 1024;
  auto kern = topk_rows_bf16_tma_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0, per_sm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 128, kSmem)) !=
      cudaSuccess)
    return e;
  const long long nblocks = (p.rows + 127) / 128;
  const long long cap = static_cast<long long>(sms) * (per_sm > 0 ? per_sm : 1);
  const unsigned grid = static_cast<unsigned>(nblocks < cap ? nblocks : cap);
  kern<<<grid, 128, kSmem, stream>>>(p.xmap, p.ymap, nblocks, p.k, p.err, p.limit_ns,
                                     p.inject_stall);
  return cudaGetLastError();
}

cudaError_t launch_topk(const TopkParams& p, cudaStream_t stream) {
  if (p.rows == 0) return cudaSuccess;
  if (p.rows > 8LL * 0x7fffffffLL) return cudaErrorInvalidValue;
  // bf16 rows up to 128 features: a thread per row (16-byte row accesses; x
  // and y are 16-byte aligned and every row is a multiple of 16 bytes)
  if (p.bf16 && p.use_tma && p.d == 128) return launch_bf16_rows_tma<128>(p, stream);
  if (p.bf16 && p.use_tma && p.d == 64) return launch_bf16_rows_tma<64>(p, stream);
  if (p.bf16 && p.d == 128) return launch_bf16_rows_staged<128>(p, stream);
  if (p.bf16 && p.d == 64) return launch_bf16_rows_staged<64>(p, stream);
  if (p.bf16 && p.d == 32) return launch_bf16_rows_staged<32>(p, stream);
  return p.bf16 ? launch_typed<__nv_bfloat16>(p, stream) : launch_typed<float>(p, stream);
}

}  // namespace spa
