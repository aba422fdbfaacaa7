// attn_ws.cu -- warp-specialised fused projected-feature attention on tcgen05
// (bf16 inputs, fp16 or split-bf16 score operands, fp32 accumulation).
//
// Persistent: one CTA per SM walks a static list of work items, each a pair
// of 128-row query tiles (t = 0, 1) of one (batch, head), streaming the
// key/value tiles of that head once for both query tiles.  Sixteen warps in
// four warpgroups (setmaxnreg moves registers from the last two to the first two):
//   warps 0-3   softmax for query tile 0   (TMEM lanes 0-127 of S0)
//   warps 4-7   softmax for query tile 1   (TMEM lanes 0-127 of S1)
//   warps 8-11  output: O_t / l for both tiles (TMEM lanes 0-127 of O0 / O1)
//   warp  12    loads: per item the two Qp tiles, then a ring of STAGES slots,
//               each a Kp tile (one bulk copy) and a V tile (TMA, 128-byte
//               swizzle) completing on one barrier
//   warp  13    tensor-memory allocation and tcgen05.mma issue
//   warps 14-15 idle (they complete the control warpgroup for the register split)
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
// shared-memory descriptor offset is a compile-time constant (each item
// starts at ring slot 0; every slot keeps its own phase bit).
//
// Between items nothing drains: the loader refills the Q tiles as soon as the
// last score MMA of the item has completed (q_empty), and the next item's
// first score MMAs follow the last PV MMAs in the same issue stream.  A
// softmax warpgroup hands its rows' max and sum to the output warpgroup
// through shared memory (stats_full[t]) and goes straight on to the next
// item's scores; the output warpgroup writes the finished O_t (o_final[t])
// through a small shared-memory staging buffer with TMA stores, and the next
// PV_t(0), which overwrites O_t, waits for o_empty[t].  (With the output on
// the softmax warpgroups, each item boundary cost them the output step:
// moving it to its own warpgroup gave C3 +2.5%, C4 m = 32 +1.6%, m = 64
// +3.3%, C5 +2.0%, bit-identical.)
//
// Online softmax (base 2, log2(e)/sqrt(m) already folded into Qp): the
// running max only moves when a tile's max exceeds it by more than 40; in
// between, probabilities up to 2^40 are accumulated (bf16 and fp32 keep the
// same relative precision at any magnitude), which leaves the final O / l
// unchanged up to rounding and skips almost every rescale of O.  The
// unnormalised O stays finite for N * 2^40 * max|v| < 2^127, i.e. for values
// below 2^(87 - log2 N) in magnitude (2^70 at N = 131072).
//
// With an `lse` buffer the output warpgroup also writes each row's log-sum-exp
// (m + log2 l, converted to natural log), which the fused backward uses to
// recompute the probabilities.
//
// Every wait is bounded (2 s).  A role that gives up sets the CTA abort flag
// and the device error word; every role leaves its loop, the MMA issuer and
// the loader wait (bounded) for their own operations in flight, the TMA stores
// finish reading shared memory, and TMEM is freed before the CTA exits.
#include <math.h>

#include "kernels.cuh"
#include "ptx.cuh"
#include "waits.cuh"

namespace spa {
namespace {

using namespace ptx;

constexpr int kThreads = 512;  // four warpgroups
// Register split.  The block is launched with 512 x 128 = 65536 registers; the
// output and control warpgroups give up part of their share to the two
// softmax warpgroups, 184 each, and keep 72 each
// (128 * (184 + 184 + 72 + 72) = 65536).  The issuer stays within 72 because
// its descriptor arithmetic is done at each MMA (opaque64/opaque32 below)
// instead of being hoisted out of the item loop.  Each warpgroup executes its
// setmaxnreg once, at the top of its branch.
struct RegSplit {
  static constexpr uint32_t kSoftmax = 184;
  static constexpr uint32_t kOutput = 72;
  static constexpr uint32_t kControl = 72;
  static_assert(128 * (2 * kSoftmax + kOutput + kControl) <= kThreads * 128,
                "register split exceeds the launch");
};
constexpr int kLoadWarp = 12;
constexpr int kMmaWarp = 13;
constexpr uint32_t kOutBar = 3;  // named barrier of the output warpgroup
// A value the compiler must treat as new at each use, so that descriptor
// arithmetic is done where the MMA is issued instead of being hoisted out of
// the item loop into registers.
__device__ __forceinline__ uint64_t opaque64(uint64_t x) {
  uint64_t r;
  asm volatile("mov.b64 %0, %1;" : "=l"(r) : "l"(x));
  return r;
}
__device__ __forceinline__ uint32_t opaque32(uint32_t x) {
  uint32_t r;
  asm volatile("mov.b32 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}
constexpr float kRescaleThreshold = 40.f;        // log2 units: p <= 2^40 between rescales
constexpr float kSumLimit = 1099511627776.f;     // 2^40: a tile row sum within it bounds every p
constexpr float kLn2 = 0.693147180559945309f;
constexpr int kBoxBytes = kTileRows * 128;  // one 128-row x 128-byte output box
constexpr int kMaxDynSmem = 227 * 1024 - 5 * 1024;  // per-block limit less the static part

template <int KD, int DV>
struct WsPlan {
  static constexpr int kStages = KD >= 128 ? 2 : 3;
  static constexpr int kQBytes = kTileRows * KD * 2;
  static constexpr int kKBytes = kTileRows * KD * 2;
  static constexpr int kVBytes = kTileRows * DV * 2;
  static constexpr int kQ = 0;                          // two Q tiles
  static constexpr int kK = 2 * kQBytes;
  static constexpr int kV = kK + kStages * kKBytes;
  static constexpr int kOps = kV + kStages * kVBytes;   // end of the operand area
  // output staging: 4, 2 or 1 boxes of 32 fp32 columns x 128 rows
  static constexpr int kBoxes = kOps + 1024 + 4 * kBoxBytes <= kMaxDynSmem   ? 4
                                : kOps + 1024 + 2 * kBoxBytes <= kMaxDynSmem ? 2
                                                                              : 1;
  static constexpr int kStage = kOps;
  static constexpr int kBytes = kStage + kBoxes * kBoxBytes;
  // one CTA per SM: a second one would wait in tcgen05.alloc for the 512 columns
  static constexpr int kLaunch = kBytes + 1024 > 120 * 1024 ? kBytes + 1024 : 120 * 1024;
  static_assert(kLaunch <= kMaxDynSmem, "shared-memory plan too large");
  static constexpr uint32_t kColsS0 = 0, kColsS1 = 128, kColsO0 = 256, kColsO1 = 256 + DV;
};

struct Bars {
  uint64_t q_full, q_empty;
  uint64_t kv_full[3], kv_empty[3];
  uint64_t s_full[2], p_full[2];
  uint64_t o_final[2], o_empty[2];
  uint64_t stats_full[2];
  uint64_t drain;
};

// Work item -> (head, query-tile pair) and the key-tile counts of its tiles.
struct Item {
  int bh, qt0, nkv0, nkv1, nkv;
};
__device__ __forceinline__ Item decode_item(const AttnTcParams& p, int w) {
  const int NT = p.NT, NP = (NT + 1) >> 1;
  // Causal work grows with the pair index, so items go out longest first
  // across all heads (pair-major); without a mask every item has the same
  // work and head-major order keeps the items that share a head's K/V together.
  Item it;
  it.bh = p.causal ? w % p.BH : w / NP;
  const int pair = NP - 1 - (p.causal ? w / p.BH : w % NP);
  it.qt0 = 2 * pair;
  const int qt1 = it.qt0 + 1;
  it.nkv0 = p.causal ? it.qt0 + 1 : NT;
  it.nkv1 = qt1 < NT ? (p.causal ? qt1 + 1 : NT) : 0;
  it.nkv = max(it.nkv0, it.nkv1);
  return it;
}
// ---------------------------------------------------------------- loader
// The loader role (one thread): per item the Qp tiles of its query-tile pair,
// then the item's key tiles through the ring of Plan::kStages slots, each slot
// a Kp tile (one bulk copy) and a V tile (TMA, 128-byte swizzle) completing on
// one barrier.  Every item starts at slot 0 and every slot keeps its own phase
// bits, so the issuer's slot numbers stay compile-time constants.  Before it
// returns, every copy it started has landed.
template <class Plan, int KD, int DV>
__device__ __forceinline__ void run_loader(const AttnTcParams& p, const CUtensorMap* vmap,
                                           uint8_t* smem, Bars& bars, const WaitCtl& ctl,
                                           int items) {
  constexpr int S = Plan::kStages;
  constexpr int kTileElems = kTileRows * KD;
  prefetch_tmap(vmap);
  uint32_t used = 0, emph = 0, armph = 0;  // per ring slot: used before, kv_empty / kv_full phase bits
  int qarmed = 0;                          // Q loads started
  bool ok = true;
  for (int k = 0; ok; ++k) {
    const int w = item_index(k, items);
    if (w < 0) break;
    const Item it = decode_item(p, w);
    if (k > 0 && !(ok = wait_or_abort(&bars.q_empty, (k - 1) & 1, ctl))) break;
    const uint16_t* Qs = p.Qs + (static_cast<size_t>(it.bh) * p.NT + it.qt0) * kTileElems;
    const uint16_t* Ks = p.Ks + static_cast<size_t>(it.bh) * p.NT * kTileElems;
    mbar_arrive_expect_tx(&bars.q_full, (it.nkv1 > 0 ? 2 : 1) * Plan::kQBytes);
    bulk_g2s(smem + Plan::kQ, Qs, Plan::kQBytes, &bars.q_full);
    if (it.nkv1 > 0)
      bulk_g2s(smem + Plan::kQ + Plan::kQBytes, Qs + kTileElems, Plan::kQBytes, &bars.q_full);
    qarmed = k + 1;
    for (int j = 0; j < it.nkv; ++j) {
      const int slot = j % S;
      const uint32_t bit = 1u << slot;
      if (used & bit) {
        if (!(ok = wait_or_abort(&bars.kv_empty[slot], (emph & bit) ? 1u : 0u, ctl)))
          break;
        emph ^= bit;
      }
      used |= bit;
      mbar_arrive_expect_tx(&bars.kv_full[slot], Plan::kKBytes + Plan::kVBytes);
      bulk_g2s(smem + Plan::kK + slot * Plan::kKBytes, Ks + static_cast<size_t>(j) * kTileElems,
               Plan::kKBytes, &bars.kv_full[slot]);
      uint8_t* vdst = smem + Plan::kV + slot * Plan::kVBytes;
#pragma unroll
      for (int h = 0; h < DV / 64; ++h)
        tma_load_3d(vdst + h * 16384, vmap, h * 64, j * kTileRows, it.bh, &bars.kv_full[slot]);
      armph ^= bit;
    }
  }
  // every copy this thread started lands before the CTA's memory is released
  // (all of them already have, unless some role gave up)
  if (qarmed > 0) mbar_wait(&bars.q_full, (qarmed - 1) & 1, ctl.limit_ns);
  for (int s = 0; s < S; ++s)
    if (used & (1u << s)) mbar_wait(&bars.kv_full[s], ((armph >> s) & 1u) ^ 1u, ctl.limit_ns);
}

// ---------------------------------------------------------------- output
// The output warpgroup writes a finished O_t / l (fp32) for query tile qt:
// DV/32 boxes of 128 rows x 128 B, staged in the 128-byte swizzle of the
// output tensor map (16-byte chunk q of row r sits at chunk q ^ (r % 8), which
// also spreads a warp's stores over all banks) through kBuffers box buffers
// at `stage` (box buffer nbox % kBuffers, nbox counting every box the
// warpgroup has written), each written out by a TMA tile store that clips rows
// past N.  The warps arrive on o_empty once their last read of O_t is done.
template <int DV, int kBuffers>
__device__ __forceinline__ void write_out_tile(uint32_t tO, uint32_t stage, int r, int lane,
                                               float inv, const CUtensorMap* omap, int qt, int bh,
                                               uint32_t bar_id, uint64_t* o_empty, int& nbox) {
  const uint32_t sw = static_cast<uint32_t>(r & 7);
#pragma unroll
  for (int b = 0; b < DV / 32; ++b) {
    uint32_t v[32];
    tmem_ld32(tO + b * 32, v);
    tmem_wait_ld();
    if (b == DV / 32 - 1) {  // O_t is read out: the next PV_t(0) may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_empty);
    }
    const uint32_t box = stage + (nbox % kBuffers) * kBoxBytes;
    ++nbox;
    if (r == 0) bulk_wait_group_read<kBuffers - 1>();  // this buffer's last store has read it
    named_bar_sync(bar_id, 128);
    const uint32_t rb = box + r * 128;
#pragma unroll
    for (int q = 0; q < 8; ++q)
      st_shared_v4(rb + ((q ^ sw) << 4), __float_as_uint(__uint_as_float(v[4 * q]) * inv),
                   __float_as_uint(__uint_as_float(v[4 * q + 1]) * inv),
                   __float_as_uint(__uint_as_float(v[4 * q + 2]) * inv),
                   __float_as_uint(__uint_as_float(v[4 * q + 3]) * inv));
    fence_proxy_async_smem();
    named_bar_sync(bar_id, 128);
    if (r == 0) {
      tma_store_3d(omap, box, b * 32, qt * kTileRows, bh);
      bulk_commit_group();
    }
  }
}

template <int KD, int DV, bool F16OPS>
__global__ void __launch_bounds__(kThreads, 1)
    attn_ws_kernel(const AttnTcParams p, const __grid_constant__ CUtensorMap vmap,
                   const __grid_constant__ CUtensorMap omap) {
  using Plan = WsPlan<KD, DV>;
  constexpr int S = Plan::kStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ Bars bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_sh;
  __shared__ float stat_l[2][2][kTileRows], stat_m[2][2][kTileRows];  // [tile][parity][row]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int items = p.BH * ((p.NT + 1) >> 1);
  const WaitCtl ctl{&abort_sh, p.err, p.limit_ns};
  // 1024-aligned operand area (128-byte swizzle atoms), as a shared-window address
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;

  if (warp == kMmaWarp) {
    tmem_alloc(&tmem_base_sh, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bars.q_full, 1);
    mbar_init(&bars.q_empty, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(&bars.kv_full[s], 1);
      mbar_init(&bars.kv_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars.s_full[t], 1);
      mbar_init(&bars.p_full[t], 4);   // one arrival per softmax warp
      mbar_init(&bars.o_final[t], 1);
      mbar_init(&bars.o_empty[t], 4);  // one arrival per output warp
      mbar_init(&bars.stats_full[t], 4);  // one arrival per softmax warp
    }
    mbar_init(&bars.drain, 1);
    abort_sh = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tmem_base_sh;
  if (warp >= 12) {
   setmaxnreg_dec<RegSplit::kControl>();  // the whole control warpgroup
   if (warp == kLoadWarp) {
    // ------------------------------------------------------------ loader
    if (lane == 0)
      run_loader<Plan, KD, DV>(p, &vmap, smem_raw + (sbase - smem_u32(smem_raw)), bars, ctl,
                               items);
   } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_f16(128, 128, F16OPS ? kFmtF16 : kFmtBF16, 0, 0);
      constexpr uint32_t kIdescPV = idesc_f16(128, DV, kFmtBF16, 0, 1);
      // descriptor bases; per-slot and per-k-step offsets below are constants
      const uint64_t dQ0 = smem_desc(sbase + Plan::kQ, 2048, 128, kLayoutInterleave);
      const uint64_t dK = smem_desc(sbase + Plan::kK, 2048, 128, kLayoutInterleave);
      const uint64_t dV = smem_desc(sbase + Plan::kV, 16384, 1024, kLayoutSwizzle128);
      bool first_s0 = true;
      auto issue_s = [&](int t, int slot) {  // S_t = Q_t K_slot^T, then signal the softmax
        const uint64_t a = opaque64(dQ0) + static_cast<uint64_t>((t * Plan::kQBytes) >> 4);
        const uint64_t b = opaque64(dK) + static_cast<uint64_t>((slot * Plan::kKBytes) >> 4);
        const uint32_t d = opaque32(tb) + (t == 0 ? Plan::kColsS0 : Plan::kColsS1);
#pragma unroll
        for (int k = 0; k < KD / 16; ++k)
          mma_ss(d, a + (k * 4096 >> 4), b + (k * 4096 >> 4), kIdescS, k > 0);
        // a failure-detection test withholds the CTA's first "S0 ready": the
        // softmax warps' wait for it runs out, and every role takes its abort path
        if (!(p.inject_stall && t == 0 && first_s0)) mma_commit(&bars.s_full[t]);
        if (t == 0) first_s0 = false;
      };
      auto issue_pv = [&](int t, int slot, uint32_t acc) {  // O_t += P_t V_slot
        const uint32_t a = opaque32(tb) + (t == 0 ? Plan::kColsS0 : Plan::kColsS1);
        const uint32_t d = opaque32(tb) + (t == 0 ? Plan::kColsO0 : Plan::kColsO1);
        const uint64_t b = opaque64(dV) + static_cast<uint64_t>((slot * Plan::kVBytes) >> 4);
        mma_ts(d, a, b, kIdescPV, acc);
#pragma unroll
        for (int k = 1; k < 8; ++k) mma_ts(d, a + k * 8, b + (k * 2048 >> 4), kIdescPV, 1u);
      };
      uint32_t fph = 0;        // per ring slot: kv_full phase bits
      uint32_t pph = 0;        // per query tile: p_full phase bits
      int ndone0 = 0, ndone1 = 0;  // items whose O_t was finished (o_final[t] committed)
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int w = item_index(k, items);
        if (w < 0) break;
        const Item it = decode_item(p, w);
        const int nkv0 = it.nkv0, nkv1 = it.nkv1, nkv = it.nkv;
        ok = wait_or_abort(&bars.q_full, k & 1, ctl) &&
             wait_or_abort(&bars.kv_full[0], fph & 1u, ctl);
        if (!ok) break;
        fph ^= 1u;
        tc_fence_after();
        issue_s(0, 0);
        if (nkv1 > 0) issue_s(1, 0);
        if (nkv == 1) mma_commit(&bars.q_empty);  // every score MMA of the item is issued
        // PV_t(0) overwrites O_t: the previous item's O_t must have been read
        // out.  Nothing else can be issued before PV0(0) anyway.
        if (ndone0 > 0 && !(ok = wait_or_abort(&bars.o_empty[0], (ndone0 - 1) & 1, ctl)))
          break;
        if (nkv1 > 0 && ndone1 > 0 &&
            !(ok = wait_or_abort(&bars.o_empty[1], (ndone1 - 1) & 1, ctl)))
          break;
        // key tiles in groups of S so that slot = u is a compile-time constant
        for (int j0 = 0; ok && j0 < nkv; j0 += S) {
#pragma unroll
          for (int u = 0; u < S; ++u) {
            const int j = j0 + u;
            if (!ok || j >= nkv) break;
            const int un = (u + 1) % S;  // slot of key tile j+1
            const bool next = j + 1 < nkv;
            if (j < nkv0) {
              if (!(ok = wait_or_abort(&bars.p_full[0], pph & 1u, ctl))) break;
              pph ^= 1u;
              tc_fence_after();
              issue_pv(0, u, j > 0 ? 1u : 0u);
            }
            if (next) {
              if (!(ok = wait_or_abort(&bars.kv_full[un], (fph >> un) & 1u, ctl))) break;
              fph ^= 1u << un;
              tc_fence_after();
              if (j + 1 < nkv0) issue_s(0, un);
            }
            if (j < nkv1) {
              if (!(ok = wait_or_abort(&bars.p_full[1], (pph >> 1) & 1u, ctl))) break;
              pph ^= 2u;
              tc_fence_after();
              issue_pv(1, u, j > 0 ? 1u : 0u);
            }
            mma_commit(&bars.kv_empty[u]);  // both tiles are done with K(j) and V(j)
            if (next && j + 1 < nkv1) issue_s(1, un);
            if (j + 2 == nkv) {
              mma_commit(&bars.q_empty);  // the item's last score MMA is issued
              // with a causal mask tile 0 ends one key tile early: finish its
              // O now, so its output overlaps tile 1's last key tile
              if (nkv0 < nkv) mma_commit(&bars.o_final[0]);
            }
          }
        }
        if (!ok) break;
        if (nkv0 == nkv) mma_commit(&bars.o_final[0]);
        if (nkv1 > 0) mma_commit(&bars.o_final[1]);
        ++ndone0;
        if (nkv1 > 0) ++ndone1;
      }
      mma_commit(&bars.drain);
      mbar_wait(&bars.drain, 0, ctl.limit_ns);  // own MMAs in flight
    }
   }  // warps 14-15: no role
  } else if (warp >= 8) {
    // ------------------------------------------------------------ output
    setmaxnreg_dec<RegSplit::kOutput>();
    const int r = tid & 127;
    const uint32_t lane_base = tb + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    int nd0 = 0, nd1 = 0, nbox = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int w = item_index(k, items);
      if (w < 0) break;
      const Item it = decode_item(p, w);
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if ((t == 0 ? it.nkv0 : it.nkv1) == 0) continue;
        const int nd = t == 0 ? nd0 : nd1;
        __syncwarp();
        ok = named_bar_and(kOutBar, 128,
                           wait_or_abort(&bars.o_final[t], nd & 1, ctl) &&
                               wait_or_abort(&bars.stats_full[t], nd & 1, ctl));
        if (!ok) break;
        tc_fence_after();
        const float l = stat_l[t][nd & 1][r], mr = stat_m[t][nd & 1][r];
        const int qt = it.qt0 + t;
        if (p.lse != nullptr) {  // log-sum-exp of the row's logits, natural log
          const int row = qt * kTileRows + r;
          if (row < p.N) p.lse[static_cast<size_t>(it.bh) * p.N + row] = (mr + log2f(l)) * kLn2;
        }
        write_out_tile<DV, Plan::kBoxes>(lane_base + (t == 0 ? Plan::kColsO0 : Plan::kColsO1),
                                         sbase + Plan::kStage, r, lane, 1.f / l, &omap, qt, it.bh,
                                         kOutBar, &bars.o_empty[t], nbox);
        if (t == 0) ++nd0; else ++nd1;
      }
    }
    if (r == 0) bulk_wait_group_read<0>();  // the stores have read shared memory
  } else {
    // ------------------------------------------------------------ softmax
    setmaxnreg_inc<RegSplit::kSoftmax>();  // the whole softmax warpgroup
    const int t = warp >> 2;  // query tile of this warpgroup
    const int r = tid & 127;  // row within the tile == TMEM lane
    const uint32_t lane_base = tb + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t tS = lane_base + (t == 0 ? Plan::kColsS0 : Plan::kColsS1);
    const uint32_t tO = lane_base + (t == 0 ? Plan::kColsO0 : Plan::kColsO1);
    uint32_t sph = 0;               // s_full phase bit
    int ndone = 0;                  // tiles whose statistics were handed over
    auto row_mul = [&](const Item& x) {
      return p.qmul[static_cast<size_t>(x.bh) * p.NT * kTileRows + (x.qt0 + t) * kTileRows + r];
    };
    for (int k = 0;; ++k) {
      const int w = item_index(k, items);
      if (w < 0) break;
      const Item it = decode_item(p, w);
      const int nkv_t = t == 0 ? it.nkv0 : it.nkv1;
      if (nkv_t == 0) continue;
      const int qt = it.qt0 + t;
      const float* kmul = p.kmul + static_cast<size_t>(it.bh) * p.NT;
      const float qm = row_mul(it);
      float m_run = -INFINITY, l_run = 0.f;
      bool ok = true;
      for (int j = 0; j < nkv_t; ++j) {
        const float km = __ldg(kmul + j);
        // warp-uniform outcome, so that the warp stays converged for the
        // .sync.aligned tensor-memory instructions below
        if (!(ok = __all_sync(0xffffffffu, wait_or_abort(&bars.s_full[t], sph, ctl))))
          break;
        sph ^= 1u;
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
        if (j == p.NT - 1) kvalid = p.N - j * kTileRows;
        if (p.causal && j == qt) kvalid = min(kvalid, r + 1);
        if (kvalid < 128) {
#pragma unroll
          for (int c = 0; c < 128; ++c) x[c] = c < kvalid ? x[c] : -INFINITY;
        }
        // The running max m_run moves only when the tile's max exceeds it by
        // more than the threshold, i.e. when some p would exceed 2^40.  So the
        // first key tile of a row takes the max, and every later one is first
        // exponentiated against m_run; only if the tile's row sum then exceeds
        // 2^40 (a sum within 2^40 bounds every term) does the warp take the
        // max and, where it moved, redo the tile from the scores still in
        // registers.  The decisions, and so the bits, are those of taking the
        // max on every tile.  With a margin of 2^20 the redo was frequent
        // where the logits spread wide (m = 16: a logit standard deviation of
        // about 11.5 in log2 units at C4, twice m = 32's), and taking the max
        // on every tile was faster there; with 2^40 the speculative form is
        // faster at every depth (C4 m = 16 +5.0%, m = 32 +0.6%, C3 +0.7%).
        const float mult = qm * km;  // > 0: range exponents times log2(e)/sqrt(m)
        float alpha = 1.f;
        bool grow = false;
        auto take_max = [&]() {  // row max: eight independent chains of three-input maxima
          float mx[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float mi = max3(x[16 * i], x[16 * i + 1], x[16 * i + 2]);
#pragma unroll
            for (int c = 3; c < 15; c += 2) mi = max3(mi, x[16 * i + c], x[16 * i + c + 1]);
            mx[i] = fmaxf(mi, x[16 * i + 15]);
          }
          const float rmax = max3(max3(mx[0], mx[1], mx[2]), max3(mx[3], mx[4], mx[5]),
                                  fmaxf(mx[6], mx[7]));
          const float tmax = rmax * mult;
          grow = tmax > m_run + kRescaleThreshold;
          if (grow) {
            alpha = ex2(m_run - tmax);  // 0 on the first tile
            m_run = tmax;
          }
        };
        // p = 2^(s * mult - m): scale and shift two at a time, exp2 on the MUFU,
        // row sum in packed pairs, bf16x2 straight into the S columns of TMEM
        auto exps = [&]() -> float {
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
          float ls = 0.f;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float a, b;
            unpack_f32x2(sum2[i], a, b);
            ls += a + b;
          }
          return ls;
        };
        if (j == 0) take_max();
        float lsum = exps();
        if (j > 0 && __any_sync(0xffffffffu, !(lsum <= kSumLimit))) {
          take_max();
          if (__any_sync(0xffffffffu, grow)) lsum = exps();  // rows that did not move: same p
        }
        // O row *= alpha when the max moved; PV(j-1) is complete (covered by the
        // S(j) commit) and PV(j) waits for p_full below.
        if (j > 0 && __any_sync(0xffffffffu, grow)) {
#pragma unroll
          for (int c0 = 0; c0 < DV; c0 += 64) {  // 64 columns per round trip
            uint32_t o0[32], o1[32];
            tmem_ld32(tO + c0, o0);
            tmem_ld32(tO + c0 + 32, o1);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              o0[i] = __float_as_uint(__uint_as_float(o0[i]) * alpha);
              o1[i] = __float_as_uint(__uint_as_float(o1[i]) * alpha);
            }
            tmem_st32(tO + c0, o0);
            tmem_st32(tO + c0 + 32, o1);
          }
        }
        l_run = l_run * alpha + lsum;
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.p_full[t]);
      }
      if (!ok) break;
      // the row's statistics for the output warpgroup, which writes O_t / l
      stat_l[t][ndone & 1][r] = l_run;
      stat_m[t][ndone & 1][r] = m_run;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.stats_full[t]);
      ++ndone;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) tmem_dealloc(tb, 512);
}

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  if (dev < 64 && cached[dev] > 0) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev < 64) cached[dev] = n;
  return n;
}

template <class Plan, class Kernel>
cudaError_t launch_persistent(Kernel kern, const AttnTcParams& p, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Plan::kLaunch);
  if (e != cudaSuccess) return e;
  const long long items = static_cast<long long>((p.NT + 1) / 2) * p.BH;
  if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
  const int sms = num_sms();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const unsigned grid = static_cast<unsigned>(items < sms ? items : sms);
  kern<<<grid, kThreads, Plan::kLaunch, stream>>>(p, p.vmap, p.omap);
  return cudaGetLastError();
}

template <int KD, int DV, bool F16OPS>
cudaError_t launch_ws(const AttnTcParams& p, cudaStream_t stream) {
  return launch_persistent<WsPlan<KD, DV>>(attn_ws_kernel<KD, DV, F16OPS>, p, stream);
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
