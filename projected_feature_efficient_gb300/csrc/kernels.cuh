// kernels.cuh -- host-side launchers shared between the C ABI (spa_api.cu)
// and the kernel translation units.  Internal to libspa.so.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace spa {

// How the projection writes its result.
enum class ProjOut : int {
  F32 = 0,       // plain fp32 rows [BH][N][m]
  F16X1 = 1,     // fp16 UMMA tiles, power-of-two row (Q) / tile (K) exponents
  BF16X3 = 2,    // bf16 hi/lo split UMMA tiles, depth 3m
  F16ROWS = 3,   // fp16 rows [BH][out_rows][m] at row out_pos + n, power-of-two row multipliers
};

// Score-GEMM operand tiles: 128 rows x KD columns of 16-bit values in the
// interleaved K-major core-matrix layout the tensor cores read directly:
//   element (r, k) of a tile sits at ((k/8)*16 + r/8)*64 + (r%8)*8 + k%8.
constexpr int kTileRows = 128;

inline int score_depth(int m, ProjOut mode) { return mode == ProjOut::BF16X3 ? 3 * m : m; }

struct ProjParams {
  const void* x[2];      // [BH][N][d] inputs (Q-like at 0, K-like at 1)
  const void* P;         // [H][d][m]
  void* out[2];          // F32: [BH][N][m] float; tiles: [BH][NT][128*KD] u16
  float* mul[2];         // tiles: Q row multipliers [BH][NT*128], K tile multipliers [BH][NT]
  int nx;                // 1 or 2 tensors
  int BH, H, N, d, m, NT;
  float qscale;          // factor folded into tensor 0 before conversion (tile modes)
  int bf16_in;           // element type of x and P: 1 = bf16, 0 = fp32
  ProjOut mode;
  int use_tc;            // tile modes: tensor-core kernel if the shape allows it
  CUtensorMap xmap[2];   // x[0], x[1] as 3-D (d, N, BH), bf16, 128-byte swizzle, box (64,128,1)
  int* err;              // device error word
  int out_rows, out_pos; // F16ROWS: rows per (batch, head) of the output, first row written
  void* out_b16[2];      // tile modes, optional: plain bf16 tiles of Xp, [BH][NT][128*m] u16
  unsigned long long limit_ns;  // tensor-core kernels: time limit of every wait (0: 2 s)
  int inject_stall;      // failure-detection test only: withhold one barrier arrival
};
bool project_tc_eligible(const ProjParams& p);
cudaError_t launch_project(const ProjParams& p, cudaStream_t stream);

struct AttnTcParams {
  const uint16_t* Qs;    // [BH][NT][128*KD]
  const uint16_t* Ks;    // [BH][NT][128*KD]
  const float* qmul;     // [BH][NT*128]
  const float* kmul;     // [BH][NT]
  CUtensorMap vmap;      // V as 3-D (d_v, N, BH), bf16, 128-byte swizzle, box (64,128,1)
  CUtensorMap omap;      // out as 3-D (d_v, N, BH), fp32, 128-byte swizzle, box (32,128,1)
  float* out;            // [BH][N][d_v]
  int* err;              // device error word
  int BH, N, NT, KD, dv, causal;
  int f16_ops;           // 1: fp16 score operands, 0: bf16
  unsigned long long limit_ns;  // time limit of every wait in the kernel
  int inject_stall;      // failure-detection test only: withhold one barrier arrival
  float* lse;            // optional [BH][N]: row log-sum-exp of the logits (natural log)
};
cudaError_t launch_attn_ws(const AttnTcParams& p, cudaStream_t stream);

struct AttnF32Params {
  const float* Qp;       // [BH][N][m]
  const float* Kp;       // [BH][N][m]
  const float* V;        // [BH][N][dv]
  float* out;            // [BH][N][dv]
  int BH, N, m, dv, causal;
  float scale;           // 1/sqrt(m)
  float* lse;            // optional [BH][N]: row log-sum-exp of the logits (natural log)
};
cudaError_t launch_attn_f32(const AttnF32Params& p, cudaStream_t stream);

// Row-wise Top-k feature sparsification: y[r] keeps the k largest-magnitude
// features of x[r] (ties: lowest feature index first) and zeroes the rest.
struct TopkParams {
  const void* x;  // [rows][d], bf16 or fp32
  void* y;        // [rows][d], same type
  long long rows;
  int d, k;       // d in {32, 64, 128, 256}, 1 <= k <= d
  int bf16;       // element type: 1 = bf16, 0 = fp32
  // bf16 rows of 64 or 128 features through TMA (when use_tma): x and y as
  // 3-D (d, rows, 1) bf16 maps, 128-byte swizzle, box (64, 128, 1)
  int use_tma;
  CUtensorMap xmap, ymap;
  int* err;       // device error word (a bounded wait that ran out)
  unsigned long long limit_ns;
  int inject_stall;  // failure-detection test only: leave one copy unissued
};
cudaError_t launch_topk(const TopkParams& p, cudaStream_t stream);
cudaError_t launch_identity(void* P, int H, int d, int bf16, cudaStream_t stream);  // P[h] = I_d

// Fused backward on tcgen05 (bf16 inputs, m in {16, 32, 64}, d_v in {64, 128}).
// Tiles are 128 rows; NT = ceil(N / 128).
struct BwdTcParams {
  const uint16_t* Qs;    // [BH][NT][128*KD] score-operand tiles, exactly the forward's
  const uint16_t* Ks;    // [BH][NT][128*KD]
  const float* kmul;     // [BH][NT] K tile range multipliers
  const uint16_t* Qb;    // [BH][NT][128*m] bf16 Qp tiles (interleaved layout)
  const uint16_t* Kb;    // [BH][NT][128*m] bf16 Kp tiles
  const float* stats;    // [BH][NT][4][128]: Q row multiplier, -lse*log2(e), -D/sqrt(m), 0
  CUtensorMap vmap;      // V  as 3-D (d_v, N, BH), bf16, 128-byte swizzle, box (64,128,1)
  CUtensorMap domap;     // dO as 3-D (d_v, N, BH), same encoding
  float* dqacc;          // [BH][NT][128*m] fp32 dQp accumulator (zeroed; tile layout of
                         // bwd_common.cuh)
  float* dkacc;          // [BH][NT][128*m] fp32 dKp, same tile layout
  float* dv_out;         // [BH][N][d_v] fp32 dV
  int* err;
  int BH, N, NT, KD, m, dv, causal;
  int f16_ops;           // 1: fp16 score operands, 0: bf16 (split) score operands
  float alpha;           // 1/sqrt(m)
  unsigned long long limit_ns;  // time limit of every wait in the kernel
  int inject_stall;      // failure-detection test only: withhold one barrier arrival
};
bool bwd_tc_supported(int m, int dv);
cudaError_t launch_bwd_tc(const BwdTcParams& p, cudaStream_t stream);
// Row statistics of the backward (persistent, TMA): dO and out as 3-D
// (d_v, N, BH) maps with 128-byte swizzle and 128-row boxes (bf16 64 columns,
// fp32 32 columns).
struct BwdStatsMaps {
  CUtensorMap domap, omap;
  int* err;                     // device error word
  unsigned long long limit_ns;  // time limit of every wait in the kernel
  int inject_stall;             // failure-detection test only: leave one copy unissued
};
cudaError_t launch_bwd_stats(const BwdStatsMaps& maps, const float* lse, const float* qmul,
                             float* stats, int BH, int N, int NT, int dv, float alpha,
                             cudaStream_t stream);
// The projection gradients in one pass on the tensor cores (d in {64, 128},
// m in {16, 32, 64}): dq = dQp P_h^T and dk = dKp P_h^T from the bf16 hi | lo
// split of the fp32 accumulators, dP_h accumulated per head in tensor memory
// and bulk-added into dP.
struct BwdFinishParams {
  CUtensorMap qmap, kmap;    // q, k as 3-D (d, N, BH), bf16, 128-byte swizzle, box (64,128,1)
  CUtensorMap dqmap, dkmap;  // dq, dk fp32 (d, N, BH), 128-byte swizzle, box (32,128,1)
  const float* dqacc;        // [BH][NT][128*m] fp32 dQp (tile layout of bwd_common.cuh)
  const float* dkacc;        // [BH][NT][128*m] fp32 dKp, same layout
  const __nv_bfloat16* P;    // [H][d][m]
  float* dP;                 // [H][d][m] fp32, zeroed by the launcher
  int* err;                  // device error word
  int B, H, N, NT, d, m;
  unsigned long long limit_ns;  // time limit of every wait in the kernel
  int inject_stall;          // failure-detection test only: withhold one barrier arrival
};
bool bwd_finish_tc_supported(int d, int m);
cudaError_t launch_bwd_finish_tc(const BwdFinishParams& p, cudaStream_t stream);

// Backward on CUDA cores for the shapes the tensor-core kernels do not cover
// (fp32 inputs; bf16 with m = 128): flash-style, the probabilities recomputed
// from the forward's row log-sum-exp, never stored; fp32 arithmetic.
struct BwdSimtParams {
  const void *q, *k, *v, *P, *dO;  // inputs (bf16 or fp32), the forward's layouts
  const float* out;                 // the forward's output [BH][N][dv]
  const float* lse;                 // the forward's row log-sum-exp [BH][N] (natural log)
  float *dq, *dk, *dv_out, *dP;     // [BH][N][d], [BH][N][d], [BH][N][dv], [H][d][m]
  float *qp, *kp, *dqp, *dkp;       // workspace: [BH][N][m] each
  float* dsum;                      // workspace: [BH][N] row sums <dO_i, O_i>
  float* part;                      // workspace: [H][chunks][d][m] partial dP
  int B, H, N, d, m, dv, causal, bf16;
  int chunks;                       // row chunks of the dP reduction
};
int bwd_simt_chunks(int B, int N);
cudaError_t launch_bwd_simt(const BwdSimtParams& p, cudaStream_t stream);

// Single-query attention against the projected key cache, split over key chunks.
constexpr int kDecodeMaxChunk = 8192;  // keys per chunk (scores in shared memory)
struct DecodeParams {
  const __nv_bfloat16* q;  // [BH][d] one query per (batch, head)
  const __nv_bfloat16* P;  // [H][d][m]
  const uint16_t* kc;      // [BH][cap][m]
  const float* kc_mul;     // [BH][cap]
  const __nv_bfloat16* v;  // [BH][cap][dv]
  float* out;              // [BH][dv]
  float* part;             // [BH][nsplit][2 + dv] chunk results (workspace)
  int BH, H, L, d, m, dv, cap, nsplit, chunk;
  float qscale;            // log2(e)/sqrt(m)
};
void decode_split(int BH, int L, int sms, int* nsplit, int* chunk);
cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream);

}  // namespace spa
