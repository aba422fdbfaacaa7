// bwd_ws.cu -- fused backward of projected-feature attention on tcgen05
// ("Sparse Projection Attention", Sec. 3.4.1: P_h is trained through the
// gradients of the attention; Algorithm 2 updates it from them).
//
// Per (batch, head), with the logits s_ij = <Qp_i, Kp_j> / sqrt(m), the
// forward's row log-sum-exp L_i and D_i = <dO_i, O_i>:
//   A_ij = exp(s_ij - L_i)                      (recomputed, never stored)
//   dV   = A^T dO
//   dS   = A * (dO V^T - D) / sqrt(m)           (gradient of Qp Kp^T)
//   dQp  = dS Kp,   dKp = dS^T Qp
// No N x N block is written to memory.  A work item is one 128-row key tile
// of one head; its CTA walks the query tiles that see it (all of them, or
// those on and below the diagonal with the causal mask), keeps dV and dKp of
// its key rows in tensor memory, and adds each query tile's share of dQp into
// an fp32 accumulator in global memory with a bulk reduce-add.
//
// Twenty-four warps in six warpgroups:
//   warps 0-15   gradient warpgroups.  TMEM lane = key row of the item's tile;
//                warpgroup g takes query columns 32g .. 32g+31.
//                  P-phase:  S^T -> P^T = exp2(S^T a_i - L_i log2 e), a_i the
//                            range multipliers of the score operands; S^T is
//                            released as soon as it is in registers, and bf16
//                            P^T goes to its own columns for the dV product.
//                  dS-phase: dP^T -> dS^T = P^T (dP^T / sqrt(m) - D_i / sqrt(m));
//                            bf16 dS^T written over its own dP^T columns (dKp
//                            product) and into a shared-memory tile in the
//                            MN-major layout the dQp product reads (dS, M = queries).
//   warps 16-19  epilogue: per query tile the column factors a_i, then the
//                dQp tile out of TMEM, through a staging tile (in slabs of at
//                most 32 columns), into the reduce-add; per item the dV rows
//                (fp32) and the dKp tile (fp32, the accumulators' tile layout).
//   warp 20      loads (one thread): per item the key tile's score operand,
//                its bf16 Kp tile and V; per query tile a two-slot ring of
//                dO, the score operand, the bf16 Qp tile and the row statistics.
//   warp 21      tensor-memory allocation; one thread issues S^T, dV and dQp.
//   warp 22      one thread issues dP^T and dKp.
//   warp 23      idle.
// Tensor memory (512 columns): S^T | dP^T/dS^T | dV | dKp | dQp | P^T, or at
// m = 64 with d_v = 128 (where that does not fit) S^T/P^T | dP^T/dS^T | dV |
// dKp | dQp with each warpgroup's P^T pairs written over its own S^T columns.
// Per query tile i the two issuing threads run
//   X: S^T(i) = Kf Qf_i^T (first tile of an item; otherwise issued early)
//      [S^T(i) in registers] S^T(i+1)      (over S^T(i))
//      [P-phase done]  dV += P^T(i) dO_i   (A from TMEM)
//      [dS-phase done] dQp_i = dS(i) Kb    (A from shared memory)
//   Y: dP^T(i) = V dO_i^T
//      [dS-phase done] dKp += dS^T(i) Qb_i (A from TMEM)
// so the scores of tile i+1 are ready when the gradient warpgroups finish
// tile i, the P-phase of tile i+1 overlaps the dKp/dQp/dP products, and the
// dS-phase of tile i overlaps the dV product.  The gradient warpgroups store
// P^T(i+1) only after the dV product of tile i has read P^T(i) (dv_done).
// MMAs from one thread execute in issue order, so an MMA that overwrites
// columns never overtakes an earlier one of the same thread reading them, and
// neither thread overwrites columns that the other one's products read.
//
// Every wait is bounded; a role that gives up sets the CTA abort flag and the
// device error word, every role leaves its loop, the issuers and the loader
// wait (bounded) for their own operations in flight, the bulk reduce-adds
// finish reading shared memory, and TMEM is freed before the CTA exits.
#include <math.h>

#include "kernels.cuh"
#include "bwd_common.cuh"
#include "ptx.cuh"
#include "waits.cuh"

namespace spa {
namespace {

using namespace ptx;

// Gradient warpgroups: each takes kGradCols of the 128 query columns of a tile.
constexpr int kGradWGs = 4;
constexpr int kGradCols = kTileRows / kGradWGs;
constexpr int kBEpiWarp = 4 * kGradWGs;         // first epilogue warp
constexpr int kBLoadWarp = kBEpiWarp + 4;
constexpr int kBMmaWarp = kBLoadWarp + 1;
constexpr int kBThreads = 32 * (kBMmaWarp + 2 + ((kBMmaWarp + 2) & 3 ? 4 - ((kBMmaWarp + 2) & 3) : 0));
// Register split: the block is launched with 768 x 80 registers; the gradient
// warpgroups give some up to the epilogue warpgroup, whose loop state and
// TMEM reads need more (the loader / issuer warpgroup keeps 80).
constexpr uint32_t kRegGrad = 72, kRegEpi = 112, kRegLaunch = 80;
static_assert(kGradWGs != 4 || 128 * (kGradWGs * kRegGrad + kRegEpi + kRegLaunch) <=
                                   kBThreads * kRegLaunch,
              "register split exceeds the launch");
// TMEM column of the bf16 pairs of queries 16 k .. 16 k + 15 (MMA k-step k) in
// a region where warpgroup g writes the pairs of its queries from column C g
__host__ __device__ constexpr uint32_t pair_col(int k) {
  return kGradCols * (16 * k / kGradCols) + 8 * (k % (kGradCols / 16));
}
constexpr int kBMaxDynSmem = 227 * 1024 - 1024;
constexpr uint32_t kEpiBar = 1;  // named barrier of the epilogue warpgroup

template <int KD, int MB, int DV>
struct BwdPlan {
  static constexpr int kKfBytes = kTileRows * KD * 2;   // score-operand tile
  static constexpr int kBBytes = kTileRows * MB * 2;    // bf16 Qp / Kp tile
  static constexpr int kVBytes = kTileRows * DV * 2;    // V or dO tile (64-column SW128 boxes)
  static constexpr int kStatBytes = 4 * kTileRows * 4;  // planes: qm, nl, dn, a
  static constexpr int kDsBytes = kTileRows * kTileRows * 2;
  // dQp leaves tensor memory in slabs of kDqSlab columns, one staging tile
  // and one bulk reduce-add each (the accumulator's tile layout, bwd_common.cuh)
  static constexpr int kDqSlab = dq_slab_cols(MB);
  static constexpr int kDqSlabs = MB / kDqSlab;
  static constexpr int kDqBytes = kTileRows * kDqSlab * 4;
  // the bf16 Qp tile is read late in a query tile (dKp product); at m = 64 it
  // is single-buffered (the next one loads during the next tile's first half)
  static constexpr int kQbStages = MB > 32 ? 1 : 2;
  // ring stage: dO | Qf | stats, padded so every dO tile is 1024-aligned
  static constexpr int kStDo = 0;
  static constexpr int kStQf = kVBytes;
  static constexpr int kStStat = kStQf + kKfBytes;
  static constexpr int kStageBytes = (kStStat + kStatBytes + 1023) / 1024 * 1024;
  static constexpr int kV = 0;
  static constexpr int kDs = kV + kVBytes;
  static constexpr int kRing = kDs + kDsBytes;
  static constexpr int kQb = kRing + 2 * kStageBytes;
  static constexpr int kKf = kQb + kQbStages * kBBytes;
  static constexpr int kKb = kKf + kKfBytes;
  static constexpr int kDq = kKb + kBBytes;
  static constexpr int kBytes = kDq + kDqBytes;
  static constexpr int kLaunch = kBytes + 1024;  // room to align the base to 1024
  static_assert(kLaunch <= kBMaxDynSmem, "backward shared-memory plan too large");
  static_assert(kVBytes % 1024 == 0 && kStageBytes % 1024 == 0, "SW128 tiles need 1024 alignment");
  // S^T | dP^T/dS^T | dV | dKp | dQp | P^T (bf16 pairs: the pair of queries
  // 2c, 2c+1 in column c, so k-step k of the dV product reads columns 8k ..).
  // Where that does not fit (m = 64 with d_v = 128), P^T is written over the
  // S^T columns of each warpgroup (k-step k reads pair_col(k)), and the next
  // S^T is issued only after the dV product has read P^T.
  static constexpr bool kPOverS = 256 + DV + 2 * MB + 64 > 512;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + DV,
                            kColDQ = 256 + DV + MB,
                            kColP = kPOverS ? 0u : 256 + DV + 2 * MB;
  static_assert(kColDQ + MB <= 512 && (kPOverS || kColP + 64 <= 512),
                "tensor-memory plan too large");
};

struct BwdBars {
  uint64_t kv_full, kv_empty;
  uint64_t qa_full[2], qa_empty[2], qb_full[2], qb_empty[2], cooked[2];
  uint64_t s_full, s_free, p_full, dp_full, ds_full, dv_done;
  uint64_t dq_full, dq_empty;
  uint64_t acc_full, acc_empty;
  uint64_t drain[2];
};

// Work item -> (head, key tile) and its query tiles qt0 .. qt0 + nq - 1.  With
// the causal mask the items go out longest first (key tile 0 sees every query
// tile) across all heads; without it, head-major so that the items sharing a
// head's queries run together.
struct BItem {
  int bh, kt, qt0, nq;
};
__device__ __forceinline__ BItem bwd_item(const BwdTcParams& p, int w) {
  BItem it;
  if (p.causal) {
    it.kt = w / p.BH;
    it.bh = w % p.BH;
    it.qt0 = it.kt;
    it.nq = p.NT - it.kt;
  } else {
    it.bh = w / p.NT;
    it.kt = w % p.NT;
    it.qt0 = 0;
    it.nq = p.NT;
  }
  return it;
}



__device__ __forceinline__ void unpack_bf16x2(uint32_t v, float& lo, float& hi) {
  lo = __uint_as_float(v << 16);
  hi = __uint_as_float(v & 0xffff0000u);
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// ---------------------------------------------------------------- loader
template <class Plan, int KD, int MB, int DV>
__device__ __forceinline__ void bwd_loader(const BwdTcParams& p, const CUtensorMap* vmap,
                                           const CUtensorMap* domap, uint8_t* smem, BwdBars& bars,
                                           const WaitCtl& ctl, int items) {
  prefetch_tmap(vmap);
  prefetch_tmap(domap);
  uint32_t g = 0;   // query tiles so far
  uint32_t ga = 0, gb = 0;  // query tiles whose part A / part B loads were started
  int karmed = 0;  // items armed so far
  bool ok = true;
  for (int k = 0; ok; ++k) {
    const int w = item_index(k, items);
    if (w < 0) break;
    const BItem it = bwd_item(p, w);
    if (k > 0 && !(ok = wait_or_abort(&bars.kv_empty, (k - 1) & 1, ctl))) break;
    const size_t ktile = static_cast<size_t>(it.bh) * p.NT + it.kt;
    mbar_arrive_expect_tx(&bars.kv_full, Plan::kKfBytes + Plan::kBBytes + Plan::kVBytes);
    bulk_g2s(smem + Plan::kKf, p.Ks + ktile * kTileRows * KD, Plan::kKfBytes, &bars.kv_full);
    bulk_g2s(smem + Plan::kKb, p.Kb + ktile * kTileRows * MB, Plan::kBBytes, &bars.kv_full);
#pragma unroll
    for (int h = 0; h < DV / 64; ++h)
      tma_load_3d(smem + Plan::kV + h * 16384, vmap, h * 64, it.kt * kTileRows, it.bh,
                  &bars.kv_full);
    karmed = k + 1;
    for (int n = 0; n < it.nq; ++n, ++g) {
      const int s = g & 1;
      // part A (dO, score operand, statistics) is free once the dV and dP^T
      // products and the gradient warps are done with it; part B (the bf16
      // Qp tile) only after the dKp product, late in the tile
      const int qt = it.qt0 + n;
      const size_t qtile = static_cast<size_t>(it.bh) * p.NT + qt;
      uint8_t* st = smem + Plan::kRing + s * Plan::kStageBytes;
      if (g >= 2 && !(ok = wait_or_abort(&bars.qa_empty[s], ((g >> 1) - 1) & 1, ctl))) break;
      mbar_arrive_expect_tx(&bars.qa_full[s], Plan::kVBytes + Plan::kKfBytes + Plan::kStatBytes);
#pragma unroll
      for (int h = 0; h < DV / 64; ++h)
        tma_load_3d(st + Plan::kStDo + h * 16384, domap, h * 64, qt * kTileRows, it.bh,
                    &bars.qa_full[s]);
      bulk_g2s(st + Plan::kStQf, p.Qs + qtile * kTileRows * KD, Plan::kKfBytes, &bars.qa_full[s]);
      bulk_g2s(st + Plan::kStStat, p.stats + qtile * 4 * kTileRows, Plan::kStatBytes,
               &bars.qa_full[s]);
      ga = g + 1;
      constexpr int QS = Plan::kQbStages;
      const int sb = QS == 2 ? s : 0;
      if (g >= QS && !(ok = wait_or_abort(&bars.qb_empty[sb], ((g / QS) - 1) & 1, ctl))) break;
      mbar_arrive_expect_tx(&bars.qb_full[sb], Plan::kBBytes);
      bulk_g2s(smem + Plan::kQb + sb * Plan::kBBytes, p.Qb + qtile * kTileRows * MB,
               Plan::kBBytes, &bars.qb_full[sb]);
      gb = g + 1;
    }
  }
  // every copy this thread started lands before the CTA's memory is released
  if (karmed > 0) mbar_wait(&bars.kv_full, (karmed - 1) & 1, ctl.limit_ns);
  for (uint32_t s = 0; s < 2; ++s) {
    const uint32_t n = ga > s ? (ga - s + 1) / 2 : 0;  // times stage s was armed
    if (n > 0) mbar_wait(&bars.qa_full[s], (n - 1) & 1, ctl.limit_ns);
  }
  constexpr uint32_t QS = Plan::kQbStages;
  for (uint32_t s = 0; s < QS; ++s) {
    const uint32_t n = gb > s ? (gb - s + QS - 1) / QS : 0;  // times Qb buffer s was armed
    if (n > 0) mbar_wait(&bars.qb_full[s], (n - 1) & 1, ctl.limit_ns);
  }
}

// ---------------------------------------------------------------- issuers
// One thread issues an unrolled run of tcgen05.mma at about 47 clocks per MMA
// when the product is small (N = 32) and at the tensor rate for N = 128; two
// threads in different warps issue side by side:
//   issuer X: S^T = Kf Qf^T, dV += P^T dO, dQp = dS Kb      (18 MMAs per tile)
//   issuer Y: dP^T = V dO^T, dKp += dS^T Qb                 (16 MMAs per tile)
// Each overwrite of tensor memory follows, in its own thread's order, the
// product that read the old contents (S^T(i+1) after dV(i) on X, dP^T(i+1)
// after dKp(i) on Y); what the two streams share goes through the gradient
// warpgroups' barriers, and each shared release (ring stage, key tile,
// accumulators) counts one commit from each issuer.
template <class Plan, int KD, int MB, int DV, bool F16OPS>
struct BwdDescs {
  static constexpr uint32_t kIdS = idesc_f16(128, 128, F16OPS ? kFmtF16 : kFmtBF16, 0, 0);
  static constexpr uint32_t kIdDP = idesc_f16(128, 128, kFmtBF16, 0, 0);
  static constexpr uint32_t kIdDV = idesc_f16(128, DV, kFmtBF16, 0, 1);
  static constexpr uint32_t kIdDK = idesc_f16(128, MB, kFmtBF16, 0, 1);
  static constexpr uint32_t kIdDQ = idesc_f16(128, MB, kFmtBF16, 1, 1);
  // K-major interleaved score operands; K-major SW128 V / dO (score-like use);
  // MN-major SW128 dO (value-like use) and dS; MN-major interleaved bf16 Qp / Kp
  uint64_t Kf, Kb, Vk, Ds, Qf[2], Qb[2], DoK[2], DoM[2];
  __device__ __forceinline__ explicit BwdDescs(uint32_t sbase) {
    Kf = smem_desc(sbase + Plan::kKf, 2048, 128, kLayoutInterleave);
    Kb = smem_desc(sbase + Plan::kKb, 128, 2048, kLayoutInterleave);
    Vk = smem_desc(sbase + Plan::kV, 16, 1024, kLayoutSwizzle128);
    Ds = smem_desc(sbase + Plan::kDs, 16384, 1024, kLayoutSwizzle128);
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const uint32_t st = sbase + Plan::kRing + s * Plan::kStageBytes;
      Qf[s] = smem_desc(st + Plan::kStQf, 2048, 128, kLayoutInterleave);
      Qb[s] = smem_desc(sbase + Plan::kQb + (s % Plan::kQbStages) * Plan::kBBytes, 128, 2048,
                        kLayoutInterleave);
      DoK[s] = smem_desc(st + Plan::kStDo, 16, 1024, kLayoutSwizzle128);
      DoM[s] = smem_desc(st + Plan::kStDo, 16384, 1024, kLayoutSwizzle128);
    }
  }
};

template <class Plan, int KD, int MB, int DV, bool F16OPS>
__device__ __forceinline__ void bwd_issuer_x(const BwdTcParams& p, uint32_t sbase, uint32_t tb,
                                             BwdBars& bars, const WaitCtl& ctl, int items) {
  using D = BwdDescs<Plan, KD, MB, DV, F16OPS>;
  const D dsc(sbase);
  bool first_s = true;
  auto issue_s = [&](int s) {  // S^T = Kf Qf^T
    const uint64_t b = s ? dsc.Qf[1] : dsc.Qf[0];
#pragma unroll
    for (int k = 0; k < KD / 16; ++k)
      mma_ss(tb + Plan::kColS, dsc.Kf + (k * 4096 >> 4), b + (k * 4096 >> 4), D::kIdS, k > 0);
    // a failure-detection test withholds the CTA's first "S^T ready": the
    // gradient warpgroups' wait for it runs out, and every role takes its abort path
    if (!(p.inject_stall && first_s)) mma_commit(&bars.s_full);
    first_s = false;
  };
  auto issue_dv = [&](int s, uint32_t acc) {  // dV += P^T dO, depth = 128 queries
    const uint64_t b = s ? dsc.DoM[1] : dsc.DoM[0];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t a = Plan::kPOverS ? Plan::kColS + pair_col(k) : Plan::kColP + 8 * k;
      mma_ts(tb + Plan::kColDV, tb + a, b + (k * 2048 >> 4), D::kIdDV, k > 0 ? 1u : acc);
    }
  };
  auto issue_dq = [&]() {  // dQp = dS Kb, depth = 128 keys
#pragma unroll
    for (int k = 0; k < 8; ++k)
      mma_ss(tb + Plan::kColDQ, dsc.Ds + (k * 2048 >> 4), dsc.Kb + (k * 256 >> 4), D::kIdDQ, k > 0);
  };
  uint32_t g = 0;  // query tiles so far
  bool ok = true;
  for (int k = 0; ok; ++k) {
    const int w = item_index(k, items);
    if (w < 0) break;
    const BItem it = bwd_item(p, w);
    if (!(ok = wait_or_abort(&bars.kv_full, k & 1, ctl))) break;
    for (int n = 0; n < it.nq; ++n, ++g) {
      const int s = g & 1;
      if (n == 0) {
        if (!(ok = wait_or_abort(&bars.qa_full[s], (g >> 1) & 1, ctl))) break;
        tc_fence_after();
        issue_s(s);
      }
      if (!Plan::kPOverS && n + 1 < it.nq) {
        // the next tile's scores as soon as the gradient warps hold S^T(i)
        // in registers: they overwrite nothing else
        const int s1 = (g + 1) & 1;
        if (!(ok = wait_or_abort(&bars.s_free, g & 1, ctl) &&
                   wait_or_abort(&bars.qa_full[s1], ((g + 1) >> 1) & 1, ctl)))
          break;
        tc_fence_after();
        issue_s(s1);
      }
      if (!(ok = wait_or_abort(&bars.p_full, g & 1, ctl))) break;
      // the first dV product of an item overwrites the accumulator: the
      // previous item's dV must have been read out
      if (n == 0 && k > 0 && !(ok = wait_or_abort(&bars.acc_empty, (k - 1) & 1, ctl))) break;
      tc_fence_after();
      issue_dv(s, n > 0 ? 1u : 0u);
      mma_commit(&bars.dv_done);     // P^T(i) is read: the P columns are free
      mma_commit(&bars.qa_empty[s]);  // X is done with part A of stage s (Qf, dO)
      if (Plan::kPOverS && n + 1 < it.nq) {
        // P^T(i) sits in the S^T columns: the next scores follow the dV
        // product that reads it, in this thread's order
        const int s1 = (g + 1) & 1;
        if (!(ok = wait_or_abort(&bars.qa_full[s1], ((g + 1) >> 1) & 1, ctl))) break;
        tc_fence_after();
        issue_s(s1);
      }
      if (!(ok = wait_or_abort(&bars.ds_full, g & 1, ctl))) break;
      if (g > 0 && !(ok = wait_or_abort(&bars.dq_empty, (g - 1) & 1, ctl))) break;
      tc_fence_after();
      issue_dq();
      mma_commit(&bars.dq_full);
    }
    if (!ok) break;
    mma_commit(&bars.kv_empty);
    mma_commit(&bars.acc_full);
  }
  mma_commit(&bars.drain[0]);
  mbar_wait(&bars.drain[0], 0, ctl.limit_ns);  // own MMAs in flight
}

template <class Plan, int KD, int MB, int DV, bool F16OPS>
__device__ __forceinline__ void bwd_issuer_y(const BwdTcParams& p, uint32_t sbase, uint32_t tb,
                                             BwdBars& bars, const WaitCtl& ctl, int items) {
  using D = BwdDescs<Plan, KD, MB, DV, F16OPS>;
  const D dsc(sbase);
  auto issue_dp = [&](int s) {  // dP^T = V dO^T, depth d_v
    const uint64_t b = s ? dsc.DoK[1] : dsc.DoK[0];
#pragma unroll
    for (int k = 0; k < DV / 16; ++k) {
      const uint32_t off = ((k >> 2) * 16384 + (k & 3) * 32) >> 4;
      mma_ss(tb + Plan::kColDP, dsc.Vk + off, b + off, D::kIdDP, k > 0);
    }
    mma_commit(&bars.dp_full);
  };
  auto issue_dk = [&](int sb, uint32_t acc) {  // dKp += dS^T Qb
    const uint64_t b = sb ? dsc.Qb[1] : dsc.Qb[0];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      mma_ts(tb + Plan::kColDK, tb + Plan::kColDP + pair_col(k), b + (k * 256 >> 4), D::kIdDK,
             k > 0 ? 1u : acc);
  };
  uint32_t g = 0;
  bool ok = true;
  for (int k = 0; ok; ++k) {
    const int w = item_index(k, items);
    if (w < 0) break;
    const BItem it = bwd_item(p, w);
    if (!(ok = wait_or_abort(&bars.kv_full, k & 1, ctl))) break;
    for (int n = 0; n < it.nq; ++n, ++g) {
      const int s = g & 1;
      if (!(ok = wait_or_abort(&bars.qa_full[s], (g >> 1) & 1, ctl))) break;
      tc_fence_after();
      issue_dp(s);  // overwrites dS^T(i-1) after dKp(i-1), in this thread's order
      mma_commit(&bars.qa_empty[s]);  // Y is done with part A of stage s (dO)
      constexpr uint32_t QS = Plan::kQbStages;
      const int sb = QS == 2 ? s : 0;
      if (!(ok = wait_or_abort(&bars.ds_full, g & 1, ctl) &&
                 wait_or_abort(&bars.qb_full[sb], (g / QS) & 1, ctl)))
        break;
      if (n == 0 && k > 0 && !(ok = wait_or_abort(&bars.acc_empty, (k - 1) & 1, ctl))) break;
      tc_fence_after();
      issue_dk(sb, n > 0 ? 1u : 0u);
      mma_commit(&bars.qb_empty[sb]);  // the bf16 Qp tile is read
    }
    if (!ok) break;
    mma_commit(&bars.kv_empty);
    mma_commit(&bars.acc_full);
  }
  mma_commit(&bars.drain[1]);
  mbar_wait(&bars.drain[1], 0, ctl.limit_ns);
}

// ---------------------------------------------------------------- gradient warpgroups
template <class Plan>
__device__ __forceinline__ void bwd_gradient(const BwdTcParams& p, uint8_t* smem, uint32_t sbase,
                                             uint32_t tb, BwdBars& bars, const WaitCtl& ctl,
                                             int items, int warp, int lane) {
  constexpr int C = kGradCols;               // query columns of this warpgroup
  constexpr int NH = C / 32;                 // 32-column TMEM loads per phase
  const int wg = warp >> 2;                 // query columns C wg .. C wg + C - 1
  const int r = (warp & 3) * 32 + lane;     // key row of the tile == TMEM lane
  const uint32_t lane_base = tb + (static_cast<uint32_t>((warp & 3) * 32) << 16);
  const uint32_t tS = lane_base + Plan::kColS + C * wg;
  // P^T pairs: in a region of their own (16 columns per warpgroup), or over
  // this warpgroup's own S^T columns
  const uint32_t tP = lane_base + (Plan::kPOverS ? Plan::kColS + C * wg : Plan::kColP + (C / 2) * wg);
  const uint32_t tDP = lane_base + Plan::kColDP + C * wg;
  // this row of the dS tile: half (C wg) / 64, first 16-byte chunk (C wg % 64) / 8
  const uint32_t srow = sbase + Plan::kDs + (C * wg / 64) * 16384 + r * 128;
  const uint32_t chunk0 = static_cast<uint32_t>((C * wg) % 64 / 8);
  const uint32_t sw = static_cast<uint32_t>(r & 7);
  const uint64_t alpha2 = pack_f32x2(p.alpha, p.alpha);
  uint32_t g = 0;
  for (int k = 0;; ++k) {
    const int w = item_index(k, items);
    if (w < 0) break;
    const BItem it = bwd_item(p, w);
    const bool row_ok = it.kt * kTileRows + r < p.N;
    bool ok = true;
    for (int n = 0; n < it.nq; ++n, ++g) {
      const int s = g & 1;
      const int qt = it.qt0 + n;
      const float* stp = reinterpret_cast<const float*>(smem + Plan::kRing + s * Plan::kStageBytes +
                                                        Plan::kStStat) + C * wg;
      // ---- P-phase: P^T = exp2(S^T a - L log2 e), masked, bf16 over S^T
      if (!(ok = __all_sync(0xffffffffu, wait_or_abort(&bars.s_full, g & 1, ctl) &&
                                             wait_or_abort(&bars.cooked[s], (g >> 1) & 1, ctl))))
        break;
      tc_fence_after();
      uint32_t x[NH][32];
#pragma unroll
      for (int h = 0; h < NH; ++h) tmem_ld32(tS + 32 * h, x[h]);
      tmem_wait_ld();
      if constexpr (!Plan::kPOverS) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.s_free);  // the next S^T may overwrite these columns
      }
      // query column c (of this warpgroup's C) is visible to key row r unless
      // the causal mask hides it on the diagonal tile; padded key rows see nothing
      const int cmin = !row_ok ? C : ((p.causal && qt == it.kt) ? r - C * wg : 0);
      uint32_t pk[NH][16];
#pragma unroll
      for (int h = 0; h < NH; ++h) {
#pragma unroll
        for (int i4 = 0; i4 < 8; ++i4) {
          const int c = 32 * h + 4 * i4;
          const float4 a4 = *reinterpret_cast<const float4*>(stp + 3 * kTileRows + c);
          const float4 l4 = *reinterpret_cast<const float4*>(stp + kTileRows + c);
          float y0, y1, y2, y3;
          unpack_f32x2(fma_f32x2(pack_f32x2(__uint_as_float(x[h][4 * i4]), __uint_as_float(x[h][4 * i4 + 1])),
                                 pack_f32x2(a4.x, a4.y), pack_f32x2(l4.x, l4.y)),
                       y0, y1);
          unpack_f32x2(fma_f32x2(pack_f32x2(__uint_as_float(x[h][4 * i4 + 2]), __uint_as_float(x[h][4 * i4 + 3])),
                                 pack_f32x2(a4.z, a4.w), pack_f32x2(l4.z, l4.w)),
                       y2, y3);
          float e0 = ex2(y0), e1 = ex2(y1), e2 = ex2(y2), e3 = ex2(y3);
          // selects without a branch (cmin = 0 keeps every value): a branch per
          // group of four kept the compiler from interleaving the groups'
          // exponentials (C4 m=32 +2.0%, C3 +0.6%, m=64 +0.8%)
          e0 = c < cmin ? 0.f : e0;
          e1 = c + 1 < cmin ? 0.f : e1;
          e2 = c + 2 < cmin ? 0.f : e2;
          e3 = c + 3 < cmin ? 0.f : e3;
          pk[h][2 * i4] = pack_bf16x2(e0, e1);
          pk[h][2 * i4 + 1] = pack_bf16x2(e2, e3);
        }
      }
      // P^T(i-1) must have been read by its dV product before P^T(i) replaces it
      if (!(ok = __all_sync(0xffffffffu, g == 0 || wait_or_abort(&bars.dv_done, (g - 1) & 1, ctl))))
        break;
      tc_fence_after();
#pragma unroll
      for (int h = 0; h < NH; ++h) tmem_st16(tP + 16 * h, pk[h]);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.p_full);

      // ---- dS-phase: dS^T = P^T (dP^T alpha - D alpha), bf16 over dP^T and into the dS tile
      if (!(ok = __all_sync(0xffffffffu,
                            wait_or_abort(&bars.dp_full, g & 1, ctl) &&
                                (g == 0 || wait_or_abort(&bars.dq_full, (g - 1) & 1, ctl)))))
        break;
      tc_fence_after();
      // dP^T 16 columns at a time (what stays live: the P pairs, the dS pairs)
      uint32_t dk[NH][16];
#pragma unroll
      for (int q16 = 0; q16 < 2 * NH; ++q16) {
        const int h = q16 >> 1, o = 8 * (q16 & 1);  // pairs o .. o + 7 of half h
        uint32_t y[16];
        tmem_ld16(tDP + 16 * q16, y);
        tmem_wait_ld();
#pragma unroll
        for (int i4 = 0; i4 < 4; ++i4) {
          const int c = 16 * q16 + 4 * i4;
          const float4 d4 = *reinterpret_cast<const float4*>(stp + 2 * kTileRows + c);
          float p0, p1, p2, p3;
          unpack_bf16x2(pk[h][o + 2 * i4], p0, p1);
          unpack_bf16x2(pk[h][o + 2 * i4 + 1], p2, p3);
          const uint64_t u01 = fma_f32x2(
              pack_f32x2(__uint_as_float(y[4 * i4]), __uint_as_float(y[4 * i4 + 1])), alpha2,
              pack_f32x2(d4.x, d4.y));
          const uint64_t u23 = fma_f32x2(
              pack_f32x2(__uint_as_float(y[4 * i4 + 2]), __uint_as_float(y[4 * i4 + 3])), alpha2,
              pack_f32x2(d4.z, d4.w));
          float s0, s1, s2, s3;
          unpack_f32x2(mul_f32x2(u01, pack_f32x2(p0, p1)), s0, s1);
          unpack_f32x2(mul_f32x2(u23, pack_f32x2(p2, p3)), s2, s3);
          dk[h][o + 2 * i4] = pack_bf16x2(s0, s1);
          dk[h][o + 2 * i4 + 1] = pack_bf16x2(s2, s3);
        }
      }
#pragma unroll
      for (int h = 0; h < NH; ++h) tmem_st16(tDP + 16 * h, dk[h]);
      // dS (M = queries) for the dQp product: 16-byte chunk q of this key row
      // holds queries 8q .. 8q + 7 of its half and sits at chunk q ^ (r % 8)
#pragma unroll
      for (int h = 0; h < NH; ++h)
#pragma unroll
        for (int j4 = 0; j4 < 4; ++j4) {
          const uint32_t q = chunk0 + 4 * h + j4;
          st_shared_v4(srow + ((q ^ sw) << 4), dk[h][4 * j4], dk[h][4 * j4 + 1], dk[h][4 * j4 + 2],
                       dk[h][4 * j4 + 3]);
        }
      fence_proxy_async_smem();
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars.ds_full);
        mbar_arrive(&bars.qa_empty[s]);  // this warp's last read of the statistics
      }
    }
    if (!ok) break;
  }
}

// ---------------------------------------------------------------- epilogue warpgroup
template <class Plan, int MB, int DV>
__device__ __forceinline__ void bwd_epilogue(const BwdTcParams& p, uint8_t* smem, uint32_t sbase,
                                             uint32_t tb, BwdBars& bars, const WaitCtl& ctl,
                                             int items, int warp, int lane) {
  const int e = (warp & 3) * 32 + lane;  // TMEM lane: query row (dQp), key row (dV, dKp)
  const uint32_t lane_base = tb + (static_cast<uint32_t>((warp & 3) * 32) << 16);
  // the accumulators' tile layout (bwd_common.cuh): slabs of W columns, chunk
  // q of row e at q ^ dsw; the staging tile holds one slab
  constexpr int W = Plan::kDqSlab;
  const uint32_t dsw = dq_slab_swizzle(e, W);
  const uint32_t stage_row = sbase + Plan::kDq + e * W * 4;

  // the column factors a_i = (Q row multiplier) x (K tile multiplier) of tile gg
  auto cook = [&](uint32_t gg, const BItem& itc) -> bool {
    const int s = gg & 1;
    if (!__all_sync(0xffffffffu, wait_or_abort(&bars.qa_full[s], (gg >> 1) & 1, ctl))) return false;
    float* stp = reinterpret_cast<float*>(smem + Plan::kRing + s * Plan::kStageBytes + Plan::kStStat);
    const float km = __ldg(p.kmul + static_cast<size_t>(itc.bh) * p.NT + itc.kt);
    stp[3 * kTileRows + e] = stp[e] * km;
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars.cooked[s]);
    return true;
  };

  int w = item_index(0, items);
  BItem it{};
  if (w >= 0) it = bwd_item(p, w);
  bool ok = w < 0 || cook(0, it);
  uint32_t g = 0;
  for (int k = 0; w >= 0; ++k) {
    const int wn = item_index(k + 1, items);
    BItem itn{};
    if (wn >= 0) itn = bwd_item(p, wn);
    for (int n = 0; n < it.nq; ++n, ++g) {
      // the next tile's column factors first: the gradient warpgroups need them
      // before this tile's dQp is even computed
      if (ok && n + 1 < it.nq) ok = cook(g + 1, it);
      else if (ok && wn >= 0) ok = cook(g + 1, itn);
      ok = ok && __all_sync(0xffffffffu, wait_or_abort(&bars.dq_full, g & 1, ctl));
      // the four warps decide together, so that they meet the barriers below as one
      if (!(ok = named_bar_and(kEpiBar, 128, ok))) break;
      tc_fence_after();
      const size_t qtile = static_cast<size_t>(it.bh) * p.NT + it.qt0 + n;
#pragma unroll
      for (int sl = 0; sl < Plan::kDqSlabs; ++sl) {
        if (e == 0) bulk_wait_group_read<0>();  // the previous reduce has read the staging tile
        named_bar_sync(kEpiBar, 128);
        // 16 columns (4 chunks) at a time: TMEM -> staging row
#pragma unroll
        for (int c16 = 0; c16 < W / 16; ++c16) {
          uint32_t v[16];
          tmem_ld16(lane_base + Plan::kColDQ + sl * W + 16 * c16, v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t q = static_cast<uint32_t>(4 * c16 + j);
            st_shared_v4(stage_row + ((q ^ dsw) << 4), v[4 * j], v[4 * j + 1], v[4 * j + 2],
                         v[4 * j + 3]);
          }
        }
        if (sl == Plan::kDqSlabs - 1) {  // dQp is read out: the next product may overwrite it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars.dq_empty);
        }
        fence_proxy_async_smem();
        named_bar_sync(kEpiBar, 128);
        if (e == 0) {
          bulk_reduce_add_f32(p.dqacc + (qtile * Plan::kDqSlabs + sl) * kTileRows * W,
                              sbase + Plan::kDq, Plan::kDqBytes);
          bulk_commit_group();
        }
      }
    }
    if (!ok) break;
    // ---- item end: dKp and dV rows of the key tile
    ok = __all_sync(0xffffffffu, wait_or_abort(&bars.acc_full, k & 1, ctl));
    if (!(ok = named_bar_and(kEpiBar, 128, ok))) break;
    tc_fence_after();
    const int row = it.kt * kTileRows + e;
    const bool wr = row < p.N;
    // dKp (fp32) into its tile of the accumulator layout, every row of the
    // tile (padded key rows hold zeros: their probabilities are masked)
    float* ktile = p.dkacc + (static_cast<size_t>(it.bh) * p.NT + it.kt) * kTileRows * MB;
#pragma unroll
    for (int c16 = 0; c16 < MB / 16; ++c16) {
      uint32_t v[16];
      tmem_ld16(lane_base + Plan::kColDK + 16 * c16, v);
      tmem_wait_ld();
      const int sl = 16 * c16 / W;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t q = static_cast<uint32_t>((16 * c16 % W) / 4 + j);
        *reinterpret_cast<float4*>(ktile + (sl * kTileRows + e) * W + ((q ^ dsw) << 2)) =
            make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                        __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
      }
    }
    float4* dvrow = reinterpret_cast<float4*>(p.dv_out + (static_cast<size_t>(it.bh) * p.N + row) * DV);
#pragma unroll
    for (int c0 = 0; c0 < DV; c0 += 16) {
      uint32_t v[16];
      tmem_ld16(lane_base + Plan::kColDV + c0, v);
      tmem_wait_ld();
      if (c0 + 16 == DV) {  // every accumulator column is read: the next item may start
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.acc_empty);
      }
      if (wr) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          dvrow[c0 / 4 + q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                          __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
      }
    }
    w = wn;
    it = itn;
  }
  if (e == 0) bulk_wait_group_read<0>();  // the reduce-adds have read shared memory
}

template <int KD, int MB, int DV, bool F16OPS>
__global__ void __launch_bounds__(kBThreads, 1)
    bwd_ws_kernel(const BwdTcParams p, const __grid_constant__ CUtensorMap vmap,
                  const __grid_constant__ CUtensorMap domap) {
  using Plan = BwdPlan<KD, MB, DV>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ BwdBars bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_sh;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int items = p.BH * p.NT;
  const WaitCtl ctl{&abort_sh, p.err, p.limit_ns};
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - smem_u32(smem_raw));

  if (warp == kBMmaWarp) {
    tmem_alloc(&tmem_base_sh, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bars.kv_full, 1);
    mbar_init(&bars.kv_empty, 2);  // one commit per issuer
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars.qa_full[s], 1);
      mbar_init(&bars.qa_empty[s], 2 + 4 * kGradWGs);  // both issuers, every gradient warp
      mbar_init(&bars.qb_full[s], 1);
      mbar_init(&bars.qb_empty[s], 1);
      mbar_init(&bars.cooked[s], 4);  // one arrival per epilogue warp
    }
    mbar_init(&bars.s_full, 1);
    mbar_init(&bars.s_free, 4 * kGradWGs);   // one arrival per gradient warp
    mbar_init(&bars.p_full, 4 * kGradWGs);
    mbar_init(&bars.dv_done, 1);
    mbar_init(&bars.dp_full, 1);
    mbar_init(&bars.ds_full, 4 * kGradWGs);
    mbar_init(&bars.dq_full, 1);
    mbar_init(&bars.dq_empty, 4);
    mbar_init(&bars.acc_full, 2);
    mbar_init(&bars.acc_empty, 4);
    mbar_init(&bars.drain[0], 1);
    mbar_init(&bars.drain[1], 1);
    abort_sh = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tmem_base_sh;
  if (warp < kBEpiWarp) {
    setmaxnreg_dec<kRegGrad>();  // every gradient warpgroup
    bwd_gradient<Plan>(p, smem, sbase, tb, bars, ctl, items, warp, lane);
  } else if (warp < kBEpiWarp + 4) {
    setmaxnreg_inc<kRegEpi>();   // the epilogue warpgroup
    bwd_epilogue<Plan, MB, DV>(p, smem, sbase, tb, bars, ctl, items, warp, lane);
  } else if (warp == kBLoadWarp) {
    if (lane == 0) bwd_loader<Plan, KD, MB, DV>(p, &vmap, &domap, smem, bars, ctl, items);
  } else if (warp == kBMmaWarp) {
    if (lane == 0) bwd_issuer_x<Plan, KD, MB, DV, F16OPS>(p, sbase, tb, bars, ctl, items);
  } else if (warp == kBMmaWarp + 1) {
    if (lane == 0) bwd_issuer_y<Plan, KD, MB, DV, F16OPS>(p, sbase, tb, bars, ctl, items);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kBMmaWarp) tmem_dealloc(tb, 512);
}

int bwd_num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

template <int KD, int MB, int DV, bool F16OPS>
cudaError_t launch_bwd(const BwdTcParams& p, cudaStream_t stream) {
  using Plan = BwdPlan<KD, MB, DV>;
  auto kern = bwd_ws_kernel<KD, MB, DV, F16OPS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Plan::kLaunch);
  if (e != cudaSuccess) return e;
  const long long items = static_cast<long long>(p.BH) * p.NT;
  if (items <= 0) return cudaSuccess;
  if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
  const int sms = bwd_num_sms();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const unsigned grid = static_cast<unsigned>(items < sms ? items : sms);
  kern<<<grid, kBThreads, Plan::kLaunch, stream>>>(p, p.vmap, p.domap);
  return cudaGetLastError();
}

template <int DV>
cudaError_t launch_bwd_dv(const BwdTcParams& p, cudaStream_t stream) {
  if (p.m == 16 && !p.f16_ops && p.KD == 48) return launch_bwd<48, 16, DV, false>(p, stream);
  if (p.m == 32 && p.f16_ops && p.KD == 32) return launch_bwd<32, 32, DV, true>(p, stream);
  if (p.m == 64 && p.f16_ops && p.KD == 64) return launch_bwd<64, 64, DV, true>(p, stream);
  return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------- small kernels
// Row statistics of the backward, stats[bh][tile][plane][r] with the planes
// (Q row multiplier, -lse log2 e, -D_i / sqrt(m), 0), D_i = <dO_i, out_i>.
// Persistent: a CTA walks (bh, 128-row tile) blocks,
// each brought in by TMA two blocks ahead through two buffers (dO as
// 64-column bf16 boxes, out as 32-column fp32 boxes, 128-byte swizzle, rows
// past N zero-filled); thread r sums row r's <dO, out> from shared memory (16-
// byte chunk c of a box row at c ^ (r % 8): a quarter warp's reads hit eight
// bank groups) and writes the tile's four statistics planes coalesced.
template <int DV>
__global__ void __launch_bounds__(128) bwd_stats_tma_kernel(
    const __grid_constant__ CUtensorMap domap, const __grid_constant__ CUtensorMap omap,
    const float* __restrict__ lse, const float* __restrict__ qmul, float* __restrict__ stats,
    int BH, int N, int NT, float alpha, int* err, unsigned long long limit_ns, int inject_stall) {
  constexpr int kBox = 128 * 128;              // one 128-row x 128-byte box
  constexpr int kDoBoxes = DV / 64, kOBoxes = DV / 32;
  constexpr int kBuf = (kDoBoxes + kOBoxes) * kBox;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[2];
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* sptr = smem_raw + (sbase - smem_u32(smem_raw));
  const int tid = threadIdx.x;
  const long long nblocks = static_cast<long long>(BH) * NT, step = gridDim.x;
  int issued0 = 0, issued1 = 0;  // thread 0: loads started into buffer 0 / 1
  auto load = [&](long long blk, int s) {
    const int bh = static_cast<int>(blk / NT), row0 = static_cast<int>(blk % NT) * kTileRows;
    mbar_arrive_expect_tx(&full[s], kBuf);
    // a failure-detection test arms CTA 0's first buffer without starting its
    // copies: the wait for it runs out, and nothing is left in flight
    if (!(inject_stall && blockIdx.x == 0 && s == 0 && issued0 == 0)) {
#pragma unroll
      for (int h = 0; h < kDoBoxes; ++h)
        tma_load_3d(sptr + s * kBuf + h * kBox, &domap, h * 64, row0, bh, &full[s]);
#pragma unroll
      for (int h = 0; h < kOBoxes; ++h)
        tma_load_3d(sptr + s * kBuf + (kDoBoxes + h) * kBox, &omap, h * 32, row0, bh, &full[s]);
    }
    if (s == 0) ++issued0;
    else ++issued1;
  };
  if (tid == 0) {
    prefetch_tmap(&domap);
    prefetch_tmap(&omap);
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
  int it = 0;
  for (long long b = b0; b < nblocks; b += step, ++it) {
    const int s = it & 1;
    ok = __syncthreads_and(mbar_wait(&full[s], (it >> 1) & 1, limit_ns));
    if (!ok) break;
    const int bh = static_cast<int>(b / NT), tile = static_cast<int>(b % NT);
    const int i = tile * kTileRows + tid;
    const uint32_t dorow = sbase + s * kBuf + tid * 128;
    const uint32_t orow = dorow + kDoBoxes * kBox;
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < DV / 8; ++c) {  // 8 columns: one dO chunk, two out chunks
      uint32_t g[4], o0[4], o1[4];
      const uint32_t cg = (c / 8) * kBox + (((c % 8) ^ sw) << 4);
      const int c0 = 2 * c, c1 = 2 * c + 1;  // out chunks (4 fp32 each)
      const uint32_t a0 = (c0 / 8) * kBox + (((c0 % 8) ^ sw) << 4);
      const uint32_t a1 = (c1 / 8) * kBox + (((c1 % 8) ^ sw) << 4);
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(g[0]), "=r"(g[1]), "=r"(g[2]), "=r"(g[3]) : "r"(dorow + cg));
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(o0[0]), "=r"(o0[1]), "=r"(o0[2]), "=r"(o0[3]) : "r"(orow + a0));
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(o1[0]), "=r"(o1[1]), "=r"(o1[2]), "=r"(o1[3]) : "r"(orow + a1));
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float lo, hi;
        unpack_bf16x2(g[e], lo, hi);
        const uint32_t* o = e < 2 ? o0 : o1;
        acc = fmaf(lo, __uint_as_float(o[(2 * e) % 4]), acc);
        acc = fmaf(hi, __uint_as_float(o[(2 * e + 1) % 4]), acc);
      }
    }
    float* st = stats + (static_cast<size_t>(bh) * NT + tile) * 4 * kTileRows + tid;
    const bool in = i < N;
    st[0] = in ? qmul[(static_cast<size_t>(bh) * NT + tile) * kTileRows + tid] : 0.f;
    st[kTileRows] = in ? -lse[static_cast<size_t>(bh) * N + i] * 1.4426950408889634f : -INFINITY;
    st[2 * kTileRows] = in ? -acc * alpha : 0.f;
    st[3 * kTileRows] = 0.f;
    // every thread has read this buffer: refill it two blocks ahead
    __syncthreads();
    if (tid == 0 && b + 2 * step < nblocks) load(b + 2 * step, s);
  }
  if (tid == 0) {
    if (!ok) atomicExch(err, 1);
    // (it iterations ran to completion: (it + 1) / 2 of them used buffer 0, it / 2 buffer 1)
    if (issued0 > (it + 1) / 2) mbar_wait(&full[0], (issued0 - 1) & 1, limit_ns);
    if (issued1 > it / 2) mbar_wait(&full[1], (issued1 - 1) & 1, limit_ns);
  }
}

}  // namespace

bool bwd_tc_supported(int m, int dv) {
  return (m == 16 || m == 32 || m == 64) && (dv == 64 || dv == 128);
}

cudaError_t launch_bwd_tc(const BwdTcParams& p, cudaStream_t stream) {
  if (p.dv == 64) return launch_bwd_dv<64>(p, stream);
  if (p.dv == 128) return launch_bwd_dv<128>(p, stream);
  return cudaErrorInvalidValue;
}

template <int DV>
cudaError_t launch_bwd_stats_tma(const BwdStatsMaps& mp, const float* lse, const float* qmul,
                                 float* stats, int BH, int N, int NT, float alpha,
                                 cudaStream_t stream) {
  constexpr int kSmem = 2 * (DV / 64 + DV / 32) * 128 * 128 + 1024;
  auto kern = bwd_stats_tma_kernel<DV>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0, per_sm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 128, kSmem)) !=
      cudaSuccess)
    return e;
  const long long nblocks = static_cast<long long>(BH) * NT;
  const long long cap = static_cast<long long>(sms) * (per_sm > 0 ? per_sm : 1);
  kern<<<static_cast<unsigned>(nblocks < cap ? nblocks : cap), 128, kSmem, stream>>>(
      mp.domap, mp.omap, lse, qmul, stats, BH, N, NT, alpha, mp.err, mp.limit_ns,
      mp.inject_stall);
  return cudaGetLastError();
}

cudaError_t launch_bwd_stats(const BwdStatsMaps& maps, const float* lse, const float* qmul,
                             float* stats, int BH, int N, int NT, int dv, float alpha,
                             cudaStream_t stream) {
  if (static_cast<long long>(BH) * NT == 0) return cudaSuccess;
  if (dv == 128) return launch_bwd_stats_tma<128>(maps, lse, qmul, stats, BH, N, NT, alpha, stream);
  if (dv == 64) return launch_bwd_stats_tma<64>(maps, lse, qmul, stats, BH, N, NT, alpha, stream);
  return cudaErrorInvalidValue;
}

}  // namespace spa
