// attn_ws.cu -- warp-specialised fused projected-feature attention on tcgen05
// (bf16 inputs, fp16 or split-bf16 score operands, fp32 accumulation).
//
// One CTA owns two 128-row query tiles (t = 0, 1) of one (batch, head) and
// streams the key/value tiles of that head once for both.  Twelve warps in
// three warpgroups (setmaxnreg moves registers from the third to the first two):
//   warps 0-3  softmax for query tile 0   (TMEM lanes 0-127 of S0 / O0)
//   warps 4-7  softmax for query tile 1   (TMEM lanes 0-127 of S1 / O1)
//   warp  8    loads: the two Qp tiles once, then a ring of STAGES slots, each
//              a Kp tile (one bulk copy) and a V tile (TMA, 128-byte swizzle)
//              completing on one barrier
//   warp  9    tensor-memory allocation and tcgen05.mma issue
//   warps 10-11 idle (they complete the control warpgroup for the register split)
// Tensor memory (512 columns):  S0 | S1 | O0 | O1, with the bf16 probabilities
// P_t written over the first 64 columns of S_t and read from there by the PV
// product.  The MMA issue order per key tile j is
//   PV0(j), S0(j+1), PV1(j), S1(j+1)
// so while one softmax warpgroup works on its tile, the tensor cores run the
// other tile's products (ping-pong).  MMAs from one thread execute in issue
// order, so S_t(j+1) never overwrites P_t(j) before PV_t(j) has read it, and
// the commit that signals "S_t(j+1) ready" also covers PV_t(j), which lets the
// softmax rescale O_t right after it without another wait.
// Issuing one tcgen05.mma costs the issuing thread about as long as a
// 128x128x16 MMA takes to execute, so the issuer does as little else as
// possible: one ring barrier per slot (not separate K and V barriers), three
// commits per key tile, and a key loop unrolled by the ring depth so every
// shared-memory descriptor offset is a compile-time constant.
//
// Online softmax (base 2, log2(e)/sqrt(m) already folded into Qp): the
// running max only moves when a tile's max exceeds it by more than 20; in
// between, probabilities up to 2^20 are accumulated (finite in bf16 and fp32,
// same relative precision), which leaves the final O / l unchanged up to
// rounding and skips almost every rescale of O.
//
// Every wait is bounded (2 s).  A role that gives up sets the CTA abort flag
// and the device error word; every role leaves its loop, the MMA issuer and
// the loader wait (bounded) for their own operations in flight, and TMEM is
// freed before the CTA exits.
#include <math.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace spa {
namespace {

using namespace ptx;

constexpr uint64_t kLimitNs = 2000000000ull;
constexpr int kThreads = 384;  // three warpgroups
// Register split.  The block is launched with 384 x 168 registers; the control
// warpgroup (warps 8-11) gives up most of its share and each softmax
// warpgroup takes 184: 128 * (184 + 184 + 128) = 63488 <= 64512.  Each
// warpgroup executes its setmaxnreg once, at the top of its branch.
constexpr uint32_t kRegsSoftmax = 184;
constexpr uint32_t kRegsControl = 128;
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
constexpr float kRescaleThreshold = 20.f;  // log2 units: p <= 2^20 between rescales

__device__ __forceinline__ uint8_t* align1k(uint8_t* p) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return reinterpret_cast<uint8_t*>((a + 1023) & ~static_cast<uintptr_t>(1023));
}

template <int KD, int DV>
struct WsPlan {
  static constexpr int kStages = KD >= 128 ? 2 : 3;
  static constexpr int kQBytes = kTileRows * KD * 2;
  static constexpr int kKBytes = kTileRows * KD * 2;
  static constexpr int kVBytes = kTileRows * DV * 2;
  static constexpr int kQ = 0;                          // two Q tiles
  static constexpr int kK = 2 * kQBytes;
  static constexpr int kV = kK + kStages * kKBytes;
  static constexpr int kBytes = kV + kStages * kVBytes;
  // one CTA per SM: a second one would wait in tcgen05.alloc for the 512 columns
  static constexpr int kLaunch = kBytes + 1024 > 120 * 1024 ? kBytes + 1024 : 120 * 1024;
  // epilogue staging of one query tile's fp32 output, reusing the Q/K/V area
  static constexpr int kStageBytes = kTileRows * DV * 4;
  static_assert(2 * kStageBytes <= kBytes, "output staging must fit in the operand area");
  static constexpr uint32_t kColsS0 = 0, kColsS1 = 128, kColsO0 = 256, kColsO1 = 256 + DV;
};

struct Bars {
  uint64_t q_full;
  uint64_t kv_full[3], kv_empty[3];
  uint64_t s_full[2], p_full[2];
  uint64_t o_final;
  uint64_t drain;
};

// Bounded wait that also gives up once another role of the CTA has aborted.
// The common case (phase already complete) costs one try_wait.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort,
                                              int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  if (*abort) return false;
  if (mbar_wait(bar, parity, kLimitNs)) return true;
  *abort = 1;
  atomicExch(err, 1);
  return false;
}

template <int KD, int DV, bool F16OPS>
__global__ void __launch_bounds__(kThreads, 1)
    attn_ws_kernel(const AttnTcParams p, const __grid_constant__ CUtensorMap vmap,
                   const __grid_constant__ CUtensorMap omap) {
  using Plan = WsPlan<KD, DV>;
  constexpr int S = Plan::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1k(smem_raw);
  __shared__ Bars bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_sh;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NT = p.NT;
  const int NP = (NT + 1) >> 1;
  // Causal work grows with the pair index, so blocks go out longest first
  // across all heads (pair-major); without a mask every block has the same
  // work and head-major order keeps the blocks that share a head's K/V together.
  const int bh = p.causal ? static_cast<int>(blockIdx.x % p.BH) : static_cast<int>(blockIdx.x / NP);
  const int pair = NP - 1 - static_cast<int>(p.causal ? blockIdx.x / p.BH : blockIdx.x % NP);
  const int qt0 = 2 * pair, qt1 = 2 * pair + 1;
  const int nkv0 = p.causal ? qt0 + 1 : NT;
  const int nkv1 = qt1 < NT ? (p.causal ? qt1 + 1 : NT) : 0;
  const int nkv = max(nkv0, nkv1);

  if (warp == kMmaWarp) {
    tmem_alloc(&tmem_base_sh, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bars.q_full, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(&bars.kv_full[s], 1);
      mbar_init(&bars.kv_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars.s_full[t], 1);
      mbar_init(&bars.p_full[t], 4);  // one arrival per softmax warp
    }
    mbar_init(&bars.o_final, 1);
    mbar_init(&bars.drain, 1);
    abort_sh = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tmem_base_sh;
  constexpr int kTileElems = kTileRows * KD;
  if (warp >= 8) {
   setmaxnreg_dec<kRegsControl>();  // the whole control warpgroup
   if (warp == kLoadWarp) {
    // ------------------------------------------------------------ loader
    if (lane == 0) {
      prefetch_tmap(&vmap);
      prefetch_tmap(&omap);
      const uint16_t* Qs = p.Qs + (static_cast<size_t>(bh) * NT + qt0) * kTileElems;
      const uint16_t* Ks = p.Ks + static_cast<size_t>(bh) * NT * kTileElems;
      mbar_arrive_expect_tx(&bars.q_full, (nkv1 > 0 ? 2 : 1) * Plan::kQBytes);
      bulk_g2s(smem + Plan::kQ, Qs, Plan::kQBytes, &bars.q_full);
      if (nkv1 > 0) bulk_g2s(smem + Plan::kQ + Plan::kQBytes, Qs + kTileElems, Plan::kQBytes,
                             &bars.q_full);
      int armed = 0;  // key tiles whose copies were started
      for (int j = 0; j < nkv; ++j) {
        const int slot = j % S;
        const uint32_t ph = (j / S) & 1;
        if (j >= S && !wait_or_abort(&bars.kv_empty[slot], ph ^ 1, &abort_sh, p.err)) break;
        mbar_arrive_expect_tx(&bars.kv_full[slot], Plan::kKBytes + Plan::kVBytes);
        bulk_g2s(smem + Plan::kK + slot * Plan::kKBytes, Ks + static_cast<size_t>(j) * kTileElems,
                 Plan::kKBytes, &bars.kv_full[slot]);
        uint8_t* vdst = smem + Plan::kV + slot * Plan::kVBytes;
#pragma unroll
        for (int h = 0; h < DV / 64; ++h)
          tma_load_3d(vdst + h * 16384, &vmap, h * 64, j * kTileRows, bh, &bars.kv_full[slot]);
        armed = j + 1;
      }
      if (abort_sh) {
        // let every copy this thread started land before the CTA's memory is reused
        mbar_wait(&bars.q_full, 0, kLimitNs);
        for (int j = max(0, armed - S); j < armed; ++j)
          mbar_wait(&bars.kv_full[j % S], (j / S) & 1, kLimitNs);
      }
    }
   } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_f16(128, 128, F16OPS ? kFmtF16 : kFmtBF16, 0, 0);
      constexpr uint32_t kIdescPV = idesc_f16(128, DV, kFmtBF16, 0, 1);
      // descriptor bases; per-slot and per-k-step offsets below are constants
      const uint64_t dQ0 = smem_desc(smem_u32(smem + Plan::kQ), 2048, 128, kLayoutInterleave);
      const uint64_t dK = smem_desc(smem_u32(smem + Plan::kK), 2048, 128, kLayoutInterleave);
      const uint64_t dV = smem_desc(smem_u32(smem + Plan::kV), 16384, 1024, kLayoutSwizzle128);
      auto issue_s = [&](int t, int slot) {  // S_t = Q_t K_slot^T, then signal the softmax
        const uint64_t a = dQ0 + static_cast<uint64_t>((t * Plan::kQBytes) >> 4);
        const uint64_t b = dK + static_cast<uint64_t>((slot * Plan::kKBytes) >> 4);
        const uint32_t d = tb + (t == 0 ? Plan::kColsS0 : Plan::kColsS1);
#pragma unroll
        for (int k = 0; k < KD / 16; ++k)
          mma_ss(d, a + (k * 4096 >> 4), b + (k * 4096 >> 4), kIdescS, k > 0);
        mma_commit(&bars.s_full[t]);
      };
      auto issue_pv = [&](int t, int slot, uint32_t acc) {  // O_t += P_t V_slot
        const uint32_t a = tb + (t == 0 ? Plan::kColsS0 : Plan::kColsS1);
        const uint32_t d = tb + (t == 0 ? Plan::kColsO0 : Plan::kColsO1);
        const uint64_t b = dV + static_cast<uint64_t>((slot * Plan::kVBytes) >> 4);
        mma_ts(d, a, b, kIdescPV, acc);
#pragma unroll
        for (int k = 1; k < 8; ++k) mma_ts(d, a + k * 8, b + (k * 2048 >> 4), kIdescPV, 1u);
      };
      bool ok = wait_or_abort(&bars.q_full, 0, &abort_sh, p.err) &&
                wait_or_abort(&bars.kv_full[0], 0, &abort_sh, p.err);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
        if (nkv1 > 0) issue_s(1, 0);
      }
      // key tiles in groups of S so that slot = u is a compile-time constant
      for (int j0 = 0; ok && j0 < nkv; j0 += S) {
#pragma unroll
        for (int u = 0; u < S; ++u) {
          const int j = j0 + u;
          if (!ok || j >= nkv) break;
          const int un = (u + 1) % S;                               // slot of key tile j+1
          const uint32_t phn = ((j0 / S) + (u + 1 == S ? 1 : 0)) & 1;  // its ring phase
          const bool next = j + 1 < nkv;
          if (j < nkv0) {
            if (!(ok = wait_or_abort(&bars.p_full[0], j & 1, &abort_sh, p.err))) break;
            tc_fence_after();
            issue_pv(0, u, j > 0 ? 1u : 0u);
          }
          if (next) {
            if (!(ok = wait_or_abort(&bars.kv_full[un], phn, &abort_sh, p.err))) break;
            tc_fence_after();
            if (j + 1 < nkv0) issue_s(0, un);
          }
          if (j < nkv1) {
            if (!(ok = wait_or_abort(&bars.p_full[1], j & 1, &abort_sh, p.err))) break;
            tc_fence_after();
            issue_pv(1, u, j > 0 ? 1u : 0u);
          }
          mma_commit(&bars.kv_empty[u]);  // both tiles are done with K(j) and V(j)
          if (next && j + 1 < nkv1) issue_s(1, un);
        }
      }
      mma_commit(ok ? &bars.o_final : &bars.drain);
      if (!ok) mbar_wait(&bars.drain, 0, kLimitNs);  // own MMAs in flight
    }
   }  // warps 10-11: no role
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    setmaxnreg_inc<kRegsSoftmax>();  // the whole softmax warpgroup
    const int t = warp >> 2;  // query tile of this warpgroup
    const int r = tid & 127;  // row within the tile == TMEM lane
    const int nkv_t = t == 0 ? nkv0 : nkv1;
    const int qt = t == 0 ? qt0 : qt1;
    const int row = qt * kTileRows + r;
    const uint32_t lane_base = tb + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t tS = lane_base + (t == 0 ? Plan::kColsS0 : Plan::kColsS1);
    const uint32_t tO = lane_base + (t == 0 ? Plan::kColsO0 : Plan::kColsO1);
    const float qm = nkv_t > 0 ? p.qmul[static_cast<size_t>(bh) * NT * kTileRows + row] : 0.f;
    const float* kmul = p.kmul + static_cast<size_t>(bh) * NT;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < nkv_t; ++j) {
      const float km = __ldg(kmul + j);
      if (!(ok = wait_or_abort(&bars.s_full[t], j & 1, &abort_sh, p.err))) break;
      tc_fence_after();
      // the whole S row: four loads in flight, one wait
      uint32_t v0[32], v1[32], v2[32], v3[32];
      tmem_ld32(tS, v0);
      tmem_ld32(tS + 32, v1);
      tmem_ld32(tS + 64, v2);
      tmem_ld32(tS + 96, v3);
      tmem_wait_ld();
      float x[128];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        x[i] = __uint_as_float(v0[i]);
        x[32 + i] = __uint_as_float(v1[i]);
        x[64 + i] = __uint_as_float(v2[i]);
        x[96 + i] = __uint_as_float(v3[i]);
      }
      // keys of this tile visible to this row
      int kvalid = 128;
      if (j == NT - 1) kvalid = p.N - j * kTileRows;
      if (p.causal && j == qt) kvalid = min(kvalid, r + 1);
      if (kvalid < 128) {
#pragma unroll
        for (int c = 0; c < 128; ++c) x[c] = c < kvalid ? x[c] : -INFINITY;
      }
      // row max: eight independent chains of three-input maxima
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float mi = max3(x[16 * i], x[16 * i + 1], x[16 * i + 2]);
#pragma unroll
        for (int k = 3; k < 15; k += 2) mi = max3(mi, x[16 * i + k], x[16 * i + k + 1]);
        mx[i] = fmaxf(mi, x[16 * i + 15]);
      }
      const float rmax = max3(max3(mx[0], mx[1], mx[2]), max3(mx[3], mx[4], mx[5]),
                              fmaxf(mx[6], mx[7]));
      const float mult = qm * km;  // > 0: range exponents times log2(e)/sqrt(m)
      const float tmax = rmax * mult;
      const bool grow = tmax > m_run + kRescaleThreshold;
      float alpha = 1.f;
      if (grow) {
        alpha = ex2(m_run - tmax);  // 0 on the first tile
        m_run = tmax;
      }
      // p = 2^(s * mult - m): scale and shift two at a time, exp2 on the MUFU,
      // row sum in packed pairs, bf16x2 straight into the S columns of TMEM
      const uint64_t mult2 = pack_f32x2(mult, mult);
      const uint64_t negm2 = pack_f32x2(-m_run, -m_run);
      uint64_t sum2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int c = h * 32 + 2 * i;
          float y0, y1;
          unpack_f32x2(fma_f32x2(pack_f32x2(x[c], x[c + 1]), mult2, negm2), y0, y1);
          const float e0 = ex2(y0), e1 = ex2(y1);
          sum2[i & 3] = add_f32x2(sum2[i & 3], pack_f32x2(e0, e1));
          pk[i] = pack_bf16x2(e0, e1);
        }
        tmem_st16(tS + h * 16, pk);
      }
      // O row *= alpha when the max moved; PV(j-1) is complete (covered by the
      // S(j) commit) and PV(j) waits for p_full below.
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
#pragma unroll
        for (int c0 = 0; c0 < DV; c0 += 64) {  // 64 columns per round trip
          uint32_t v0[32], v1[32];
          tmem_ld32(tO + c0, v0);
          tmem_ld32(tO + c0 + 32, v1);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            v0[i] = __float_as_uint(__uint_as_float(v0[i]) * alpha);
            v1[i] = __float_as_uint(__uint_as_float(v1[i]) * alpha);
          }
          tmem_st32(tO + c0, v0);
          tmem_st32(tO + c0 + 32, v1);
        }
      }
      float lsum = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float a, b;
        unpack_f32x2(sum2[i], a, b);
        lsum += a + b;
      }
      l_run = l_run * alpha + lsum;
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.p_full[t]);
    }
    // epilogue: O / l -> out (fp32), staged in shared memory and written by
    // TMA stores.  Once o_final has fired every MMA is complete and every load
    // consumed, so tile t stages its 128 x DV block over the operand area at
    // t * kStageBytes, as DV/32 boxes of 128 rows x 128 B in the 128-byte
    // swizzle of the output tensor map (16-byte chunk q of row r sits at chunk
    // q ^ (r % 8)), which also spreads a warp's stores over all banks.  The
    // store clips rows past N.  All 128 threads of the warpgroup reach the
    // named barrier; a thread that gave up has set abort_sh before it.
    if (nkv_t > 0) {
      const uint32_t stage_base = ((smem_u32(smem_raw) + 1023u) & ~1023u) + t * Plan::kStageBytes;
      if (ok && wait_or_abort(&bars.o_final, 0, &abort_sh, p.err)) {
        tc_fence_after();
        const float inv = 1.f / l_run;
        const uint32_t row_base = stage_base + r * 128;
        const uint32_t sw = static_cast<uint32_t>(r & 7);
#pragma unroll
        for (int c0 = 0; c0 < DV; c0 += 32) {
          uint32_t v[32];
          tmem_ld32(tO + c0, v);
          tmem_wait_ld();
          const uint32_t rb = row_base + (c0 / 32) * (kTileRows * 128);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            st_shared_v4(rb + ((q ^ sw) << 4),
                         __float_as_uint(__uint_as_float(v[4 * q]) * inv),
                         __float_as_uint(__uint_as_float(v[4 * q + 1]) * inv),
                         __float_as_uint(__uint_as_float(v[4 * q + 2]) * inv),
                         __float_as_uint(__uint_as_float(v[4 * q + 3]) * inv));
        }
        fence_proxy_async_smem();
      }
      if (t == 0) named_bar_sync(1, 128); else named_bar_sync(2, 128);
      if (r == 0 && !abort_sh) {
#pragma unroll
        for (int c0 = 0; c0 < DV; c0 += 32)
          tma_store_3d(&omap, stage_base + (c0 / 32) * (kTileRows * 128), c0, qt * kTileRows, bh);
        bulk_commit_group();
        bulk_wait_group_read0();
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) tmem_dealloc(tb, 512);
}

template <int KD, int DV, bool F16OPS>
cudaError_t launch_ws(const AttnTcParams& p, cudaStream_t stream) {
  using Plan = WsPlan<KD, DV>;
  auto kern = attn_ws_kernel<KD, DV, F16OPS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Plan::kLaunch);
  if (e != cudaSuccess) return e;
  const long long blocks = static_cast<long long>((p.NT + 1) / 2) * p.BH;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  kern<<<static_cast<unsigned>(blocks), kThreads, Plan::kLaunch, stream>>>(p, p.vmap, p.omap);
  return cudaGetLastError();
}

template <int DV>
cudaError_t launch_ws_dv(const AttnTcParams& p, cudaStream_t stream) {
  if (!p.f16_ops) {
    if (p.KD == 48) return launch_ws<48, DV, false>(p, stream);
    return cudaErrorInvalidValue;
  }
  switch (p.KD) {
    case 32: return launch_ws<32, DV, true>(p, stream);
    case 64: return launch_ws<64, DV, true>(p, stream);
    case 128: return launch_ws<128, DV, true>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_attn_ws(const AttnTcParams& p, cudaStream_t stream) {
  if (p.dv == 64) return launch_ws_dv<64>(p, stream);
  if (p.dv == 128) return launch_ws_dv<128>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace spa
