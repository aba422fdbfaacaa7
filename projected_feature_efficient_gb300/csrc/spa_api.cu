// spa_api.cu -- the C ABI of libspa.so (declared in include/spa.h): argument
// validation, workspace layout, tensor-map encoding, launches and status codes.
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "../../include/spa.h"
#include "kernels.cuh"

namespace {

using spa::ProjOut;

// Device word set by a kernel that gave up on a bounded wait.
__device__ int g_spa_device_error;

constexpr int kMaxDevices = 64;
int* g_err_ptr[kMaxDevices] = {};
std::mutex g_err_mu;

int device_error_ptr(int** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_err_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_spa_device_error) != cudaSuccess) return SPA_ERR_CUDA;
    g_err_ptr[dev] = static_cast<int*>(p);
  }
  *out = g_err_ptr[dev];
  return SPA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

int get_encode(PFN_cuTensorMapEncodeTiled_v12000* fn) {
  std::call_once(g_encode_once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  *fn = g_encode;
  return g_encode ? SPA_OK : SPA_ERR_CUDA;
}

constexpr int kEmpty = -1;  // internal: nothing to do

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape / dtype checks shared by every forward entry point.
int check_shape(int B, int H, int N, int d, int m, int dv, int dtype) {
  if (B < 0 || H < 0 || N < 0 || d < 0 || m < 0 || dv < 0) return SPA_ERR_SHAPE;
  if (dtype != SPA_F32 && dtype != SPA_BF16) return SPA_ERR_DTYPE;
  if (static_cast<long long>(B) * H * N == 0) return kEmpty;
  if (static_cast<long long>(B) * H > 65535) return SPA_ERR_SHAPE;
  if (d < 1 || d > 256 || m < 1 || m > 128 || dv < 1 || dv > 256) return SPA_ERR_UNSUPPORTED;
  if (dtype == SPA_BF16) {
    if (m != 16 && m != 32 && m != 64 && m != 128) return SPA_ERR_UNSUPPORTED;
    if (dv != 64 && dv != 128) return SPA_ERR_UNSUPPORTED;
  }
  return SPA_OK;
}

struct Layout {
  int NT = 0, KD = 0;
  ProjOut mode = ProjOut::F32;
  size_t qs = 0, ks = 0, qmul = 0, kmul = 0;  // bf16 path
  size_t qp = 0, kp = 0;                      // fp32 path
  size_t total = 0;
};

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

Layout make_layout(int B, int H, int N, int m, int dtype) {
  Layout L;
  const size_t BH = static_cast<size_t>(B) * H;
  if (dtype == SPA_BF16) {
    L.NT = (N + spa::kTileRows - 1) / spa::kTileRows;
    L.mode = m == 16 ? ProjOut::BF16X3 : ProjOut::F16X1;
    L.KD = spa::score_depth(m, L.mode);
    const size_t tiles = BH * L.NT * spa::kTileRows * L.KD * 2;
    L.qs = 0;
    L.ks = align256(L.qs + tiles);
    L.qmul = align256(L.ks + tiles);
    L.kmul = align256(L.qmul + BH * L.NT * spa::kTileRows * sizeof(float));
    L.total = align256(L.kmul + BH * L.NT * sizeof(float));
  } else {
    const size_t proj = BH * N * m * sizeof(float);
    L.qp = 0;
    L.kp = align256(proj);
    L.total = align256(L.kp + proj);
  }
  return L;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? SPA_OK : SPA_ERR_CUDA; }

spa::ProjParams proj_params(const void* q, const void* k, const void* P, int B, int H, int N,
                            int d, int m, int dtype, const Layout& L, char* w) {
  spa::ProjParams pp{};
  pp.x[0] = q;
  pp.x[1] = k;
  pp.P = P;
  pp.nx = 2;
  pp.BH = B * H;
  pp.H = H;
  pp.N = N;
  pp.d = d;
  pp.m = m;
  pp.bf16_in = dtype == SPA_BF16;
  pp.NT = (N + spa::kTileRows - 1) / spa::kTileRows;
  if (dtype == SPA_F32) {
    pp.mode = ProjOut::F32;
    pp.out[0] = w + L.qp;
    pp.out[1] = w + L.kp;
  } else {
    pp.mode = L.mode;
    pp.out[0] = w + L.qs;
    pp.out[1] = w + L.ks;
    pp.mul[0] = reinterpret_cast<float*>(w + L.qmul);
    pp.mul[1] = reinterpret_cast<float*>(w + L.kmul);
    // scores come out in base-2 logits: fold log2(e) / sqrt(m) into Q
    pp.qscale = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(m)));
  }
  return pp;
}

// Row-major [BH][N][inner] tensor as a 3-D tensor map with 128-byte swizzle and
// 128-row boxes whose inner extent is 128 bytes (64 bf16 or 32 fp32 values).
int encode_rows_map(CUtensorMap* map, const void* base, int inner, int N, int BH,
                    CUtensorMapDataType type, int elem_bytes) {
  PFN_cuTensorMapEncodeTiled_v12000 encode;
  int st = get_encode(&encode);
  if (st) return st;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner) * elem_bytes,
                           static_cast<cuuint64_t>(N) * inner * elem_bytes};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / elem_bytes),
                       static_cast<cuuint32_t>(spa::kTileRows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  if (encode(map, type, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return SPA_ERR_CUDA;
  return SPA_OK;
}
int encode_bf16_rows(CUtensorMap* map, const void* base, int inner, int N, int BH) {
  return encode_rows_map(map, base, inner, N, BH, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2);
}

// Stage 1: projection of q and k into the workspace (and, for the backward,
// plain bf16 tiles of Qp and Kp into qb, kb in the same pass).
int run_prepare(const void* q, const void* k, const void* P, int B, int H, int N, int d, int m,
                int dtype, void* ws, cudaStream_t stream, void* qb = nullptr, void* kb = nullptr,
                unsigned long long limit_ns = 0, int inject_stall = 0) {
  const Layout L = make_layout(B, H, N, m, dtype);
  spa::ProjParams pp = proj_params(q, k, P, B, H, N, d, m, dtype, L, static_cast<char*>(ws));
  pp.use_tc = 1;
  pp.out_b16[0] = qb;
  pp.out_b16[1] = kb;
  pp.limit_ns = limit_ns;
  pp.inject_stall = inject_stall;
  if (spa::project_tc_eligible(pp)) {
    int st;
    if ((st = encode_bf16_rows(&pp.xmap[0], q, d, N, B * H))) return st;
    if ((st = encode_bf16_rows(&pp.xmap[1], k, d, N, B * H))) return st;
    if ((st = device_error_ptr(&pp.err))) return st;
  }
  return cuda_status(spa::launch_project(pp, stream));
}

// Stage 2: scores, mask, online softmax and the value product from a prepared workspace.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s per wait

int run_apply(const void* v, float* out, int B, int H, int N, int m, int dv, int causal,
              int dtype, const void* ws, cudaStream_t stream,
              unsigned long long limit_ns = kWaitLimitNs, int inject_stall = 0,
              float* lse = nullptr) {
  const Layout L = make_layout(B, H, N, m, dtype);
  const int BH = B * H;
  const char* w = static_cast<const char*>(ws);
  if (dtype == SPA_F32) {
    spa::AttnF32Params ap{};
    ap.Qp = reinterpret_cast<const float*>(w + L.qp);
    ap.Kp = reinterpret_cast<const float*>(w + L.kp);
    ap.V = static_cast<const float*>(v);
    ap.out = out;
    ap.BH = BH;
    ap.N = N;
    ap.m = m;
    ap.dv = dv;
    ap.causal = causal != 0;
    ap.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(m)));
    ap.lse = lse;
    return cuda_status(spa::launch_attn_f32(ap, stream));
  }
  int st;
  spa::AttnTcParams ap{};
  if ((st = encode_bf16_rows(&ap.vmap, v, dv, N, BH))) return st;
  if ((st = encode_rows_map(&ap.omap, out, dv, N, BH, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4)))
    return st;
  int* err = nullptr;
  if ((st = device_error_ptr(&err))) return st;
  ap.Qs = reinterpret_cast<const uint16_t*>(w + L.qs);
  ap.Ks = reinterpret_cast<const uint16_t*>(w + L.ks);
  ap.qmul = reinterpret_cast<const float*>(w + L.qmul);
  ap.kmul = reinterpret_cast<const float*>(w + L.kmul);
  ap.out = out;
  ap.err = err;
  ap.BH = BH;
  ap.N = N;
  ap.NT = L.NT;
  ap.KD = L.KD;
  ap.dv = dv;
  ap.causal = causal != 0;
  ap.f16_ops = L.mode == ProjOut::F16X1;
  ap.limit_ns = limit_ns;
  ap.inject_stall = inject_stall;
  ap.lse = lse;
  return cuda_status(spa::launch_attn_ws(ap, stream));
}

int run_forward(const void* q, const void* k, const void* v, const void* P, float* out, int B,
                int H, int N, int d, int m, int dv, int causal, int dtype, void* ws,
                cudaStream_t stream) {
  int st = run_prepare(q, k, P, B, H, N, d, m, dtype, ws, stream);
  if (st) return st;
  return run_apply(v, out, B, H, N, m, dv, causal, dtype, ws, stream);
}

int check_forward_ptrs(const void* q, const void* k, const void* v, const void* P,
                       const void* out) {
  if (!q || !k || !v || !P || !out) return SPA_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(P) || !aligned16(out))
    return SPA_ERR_ALIGN;
  return SPA_OK;
}

}  // namespace

namespace {

// Host-buffer forward, pipelined over chunks of whole heads of one batch
// entry: chunk c is copied in, projected, attended and copied out on stream
// slot c % kHostSlots, so the copy engines bring chunk c+1 in and take chunk
// c-1 out while chunk c computes.  Heads are independent, and a chunk of heads
// [h0, h0+n) of batch entry b is the problem (B=1, H=n) on the matching slices
// of q, k, v, out and P.
constexpr int kHostSlots = 4;

// The host-buffer forward's device staging comes from a pool of the library's
// own, one per device, which keeps what it has reserved between calls (the
// default pool hands memory back to the driver at every synchronisation, and
// reserving a few GB again costs more than the copies it stages).
cudaMemPool_t g_host_pool[kMaxDevices] = {};
std::mutex g_host_pool_mu;

int host_pool(cudaMemPool_t* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_host_pool_mu);
  if (!g_host_pool[dev]) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool = nullptr;
    if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) {
      cudaGetLastError();
      return SPA_ERR_CUDA;
    }
    uint64_t keep = UINT64_MAX;
    if (cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess) {
      cudaGetLastError();
      cudaMemPoolDestroy(pool);
      return SPA_ERR_CUDA;
    }
    g_host_pool[dev] = pool;
  }
  *out = g_host_pool[dev];
  return SPA_OK;
}
// Stream-ordered workspace from the library's pool: it keeps what it has
// reserved across synchronisations, so calls in a synchronised loop do not
// reserve device memory again (with the default pool, which hands memory back
// at every synchronisation, the allocating forward took 0.64 ms per call on C3
// against 0.36 ms on a caller workspace).  Released with cudaFreeAsync.
int pool_alloc(void** p, size_t bytes, cudaStream_t s) {
  cudaMemPool_t pool = nullptr;
  if (host_pool(&pool) != SPA_OK) return SPA_ERR_CUDA;
  if (cudaMallocFromPoolAsync(p, bytes, pool, s) != cudaSuccess) {
    cudaGetLastError();
    return SPA_ERR_NOMEM;
  }
  return SPA_OK;
}

// The host-buffer forward's internal streams, created once per device and kept
// until the process exits (creating and destroying them took about 0.05 ms of
// every call).  Calls from several threads may share them: each call orders
// its chunks after its own stream with its own events, so sharing only adds
// ordering between calls.
cudaStream_t g_host_streams[kMaxDevices][kHostSlots] = {};

int host_streams(cudaStream_t (&out)[kHostSlots]) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_host_pool_mu);
  for (int j = 0; j < kHostSlots; ++j) {
    if (!g_host_streams[dev][j] &&
        cudaStreamCreateWithFlags(&g_host_streams[dev][j], cudaStreamNonBlocking) != cudaSuccess) {
      cudaGetLastError();
      g_host_streams[dev][j] = nullptr;
      return SPA_ERR_CUDA;
    }
    out[j] = g_host_streams[dev][j];
  }
  return SPA_OK;
}
constexpr size_t kHostChunkBytes = size_t(32) << 20;  // aim for at least this per chunk
// at most this many chunks (C4 shape: one head per chunk; measured on GB300,
// four slots and up to 32 chunks 8.81 ms per forward, three slots and 16
// chunks 9.13 ms)
constexpr int kHostMaxChunks = 32;

int host_forward(const char* q, const char* k, const char* v, const char* P, float* out, int B,
                 int H, int N, int d, int m, int dv, int causal, int dtype, cudaStream_t stream) {
  const size_t es = dtype == SPA_BF16 ? 2 : 4;
  const size_t head_in = static_cast<size_t>(N) * (2 * d + dv) * es;
  const size_t head_out = static_cast<size_t>(N) * dv * sizeof(float);
  const size_t total_heads = static_cast<size_t>(B) * H;
  const size_t want = (total_heads * (head_in + head_out)) / kHostChunkBytes;
  const size_t nchunks = want < 1 ? 1 : (want > kHostMaxChunks ? kHostMaxChunks : want);
  size_t per = (total_heads + nchunks - 1) / nchunks;
  const int nh = static_cast<int>(per < 1 ? 1 : (per > static_cast<size_t>(H) ? H : per));

  // one slot: q, k, v, P slices, out slice and the workspace for nh heads
  const size_t nq = static_cast<size_t>(nh) * N * d * es, nv = static_cast<size_t>(nh) * N * dv * es;
  const size_t np = static_cast<size_t>(nh) * d * m * es, no = static_cast<size_t>(nh) * N * dv * 4;
  const size_t oq = 0, ok = align256(oq + nq), ov = align256(ok + nq), op = align256(ov + nv),
               oo = align256(op + np), ow = align256(oo + no);
  const size_t slot_bytes = align256(ow + make_layout(1, nh, N, m, dtype).total);

  cudaStream_t ss[kHostSlots] = {};
  cudaEvent_t ev_begin = nullptr, ev_end[kHostSlots] = {};
  char* dbuf = nullptr;
  int st = SPA_OK;
  auto fail = [&](cudaError_t e) {
    if (e != cudaSuccess && st == SPA_OK) st = SPA_ERR_CUDA;
    return e != cudaSuccess;
  };
  cudaMemPool_t pool = nullptr;
  if (host_pool(&pool) != SPA_OK || host_streams(ss) != SPA_OK) return SPA_ERR_CUDA;
  if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&dbuf), kHostSlots * slot_bytes, pool,
                              stream) != cudaSuccess) {
    cudaGetLastError();
    return SPA_ERR_NOMEM;
  }
  bool ready = !fail(cudaEventCreateWithFlags(&ev_begin, cudaEventDisableTiming)) &&
               !fail(cudaEventRecord(ev_begin, stream));
  for (int j = 0; ready && j < kHostSlots; ++j)
    ready = !fail(cudaEventCreateWithFlags(&ev_end[j], cudaEventDisableTiming)) &&
            !fail(cudaStreamWaitEvent(ss[j], ev_begin, 0));
  int c = 0;
  for (int b = 0; ready && st == SPA_OK && b < B; ++b) {
    for (int h0 = 0; st == SPA_OK && h0 < H; h0 += nh, ++c) {
      const int n = H - h0 < nh ? H - h0 : nh;
      cudaStream_t sj = ss[c % kHostSlots];
      char* sb = dbuf + (c % kHostSlots) * slot_bytes;
      const size_t head0 = static_cast<size_t>(b) * H + h0;
      const size_t cq = static_cast<size_t>(n) * N * d * es, cv = static_cast<size_t>(n) * N * dv * es;
      if (fail(cudaMemcpyAsync(sb + oq, q + head0 * N * d * es, cq, cudaMemcpyHostToDevice, sj)) ||
          fail(cudaMemcpyAsync(sb + ok, k + head0 * N * d * es, cq, cudaMemcpyHostToDevice, sj)) ||
          fail(cudaMemcpyAsync(sb + ov, v + head0 * N * dv * es, cv, cudaMemcpyHostToDevice, sj)) ||
          fail(cudaMemcpyAsync(sb + op, P + static_cast<size_t>(h0) * d * m * es,
                               static_cast<size_t>(n) * d * m * es, cudaMemcpyHostToDevice, sj)))
        break;
      st = run_forward(sb + oq, sb + ok, sb + ov, sb + op, reinterpret_cast<float*>(sb + oo), 1, n,
                       N, d, m, dv, causal, dtype, sb + ow, sj);
      if (st) break;
      if (fail(cudaMemcpyAsync(out + head0 * N * dv, sb + oo, static_cast<size_t>(n) * N * dv * 4,
                               cudaMemcpyDeviceToHost, sj)))
        break;
    }
  }
  // join every slot back into the caller's stream, release, and wait
  for (int j = 0; j < kHostSlots; ++j)
    if (ss[j] && ev_end[j] && !fail(cudaEventRecord(ev_end[j], ss[j])))
      fail(cudaStreamWaitEvent(stream, ev_end[j], 0));
  fail(cudaFreeAsync(dbuf, stream));
  fail(cudaStreamSynchronize(stream));
  for (int j = 0; j < kHostSlots; ++j)
    if (ev_end[j]) cudaEventDestroy(ev_end[j]);
  if (ev_begin) cudaEventDestroy(ev_begin);
  return st;
}

// ---------------------------------------------------------------- fused backward
// Workspace of the fused backward: the forward's prepared operands (so that
// the recomputed scores are bit-identical to the forward's), bf16 Qp / Kp
// tiles for the gradient products, the row statistics, the fp32 dQp and dKp
// accumulators (tile layout of bwd_common.cuh), and (when the caller has no
// log-sum-exp) lse plus a scratch output.
struct BwdLayout {
  Layout fwd;
  size_t qb = 0, kb = 0, stats = 0, dqacc = 0, dkacc = 0;
  size_t lse = 0, out2 = 0, total = 0;
};

BwdLayout make_bwd_layout(int B, int H, int N, int d, int m, int dv, bool own_lse) {
  BwdLayout L;
  L.fwd = make_layout(B, H, N, m, SPA_BF16);
  const size_t BH = static_cast<size_t>(B) * H, rows = BH * L.fwd.NT * spa::kTileRows;
  size_t o = L.fwd.total;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  L.qb = take(rows * m * 2);
  L.kb = take(rows * m * 2);
  L.stats = take(rows * 4 * sizeof(float));
  L.dqacc = take(rows * m * sizeof(float));
  L.dkacc = take(rows * m * sizeof(float));
  if (own_lse) {
    L.lse = take(BH * N * sizeof(float));
    L.out2 = take(BH * N * dv * sizeof(float));
  }
  L.total = o;
  return L;
}

// The tensor-core backward (fused kernel and one-pass finish); every other
// shape runs on CUDA cores (run_backward_simt).
bool bwd_fused_eligible(int d, int m, int dv, int dtype) {
  return dtype == SPA_BF16 && spa::bwd_tc_supported(m, dv) && spa::bwd_finish_tc_supported(d, m);
}

// Fused backward, stage 1 on a workspace laid out by make_bwd_layout, after
// run_prepare (given the layout's qb / kb) has put the forward's score operands
// and the bf16 Qp / Kp tiles in it: the zeroed dQp accumulator and the row
// statistics.
int bwd_stage_inputs(const float* out, const float* lse, const void* dO, int B, int H, int N,
                     int d, int m, int d_v, char* w, cudaStream_t stream,
                     unsigned long long limit_ns = kWaitLimitNs, int inject_stall = 0) {
  const BwdLayout L = make_bwd_layout(B, H, N, d, m, d_v, false);
  const int BH = B * H, NT = L.fwd.NT;
  int st;
  const float alpha = static_cast<float>(1.0 / std::sqrt(static_cast<double>(m)));
  if ((st = cuda_status(cudaMemsetAsync(w + L.dqacc, 0,
                                        static_cast<size_t>(BH) * NT * spa::kTileRows * m *
                                            sizeof(float),
                                        stream))))
    return st;
  spa::BwdStatsMaps maps{};
  if ((st = encode_bf16_rows(&maps.domap, dO, d_v, N, BH)) ||
      (st = encode_rows_map(&maps.omap, out, d_v, N, BH, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4)) ||
      (st = device_error_ptr(&maps.err)))
    return st;
  maps.limit_ns = limit_ns;
  maps.inject_stall = inject_stall;
  return cuda_status(spa::launch_bwd_stats(
      maps, lse, reinterpret_cast<const float*>(w + L.fwd.qmul),
      reinterpret_cast<float*>(w + L.stats), BH, N, NT, d_v, alpha, stream));
}

// Fused backward, stage 2: the tensor-core kernel (dV, dKp, dQp).
int bwd_stage_kernel(const void* v, const void* dO, float* dv, int B, int H, int N, int d, int m,
                     int d_v, int causal, char* w, cudaStream_t stream,
                     unsigned long long limit_ns = kWaitLimitNs, int inject_stall = 0) {
  const BwdLayout L = make_bwd_layout(B, H, N, d, m, d_v, false);
  const int BH = B * H;
  int st;
  spa::BwdTcParams bp{};
  if ((st = encode_bf16_rows(&bp.vmap, v, d_v, N, BH))) return st;
  if ((st = encode_bf16_rows(&bp.domap, dO, d_v, N, BH))) return st;
  if ((st = device_error_ptr(&bp.err))) return st;
  bp.Qs = reinterpret_cast<const uint16_t*>(w + L.fwd.qs);
  bp.Ks = reinterpret_cast<const uint16_t*>(w + L.fwd.ks);
  bp.kmul = reinterpret_cast<const float*>(w + L.fwd.kmul);
  bp.Qb = reinterpret_cast<const uint16_t*>(w + L.qb);
  bp.Kb = reinterpret_cast<const uint16_t*>(w + L.kb);
  bp.stats = reinterpret_cast<const float*>(w + L.stats);
  bp.dqacc = reinterpret_cast<float*>(w + L.dqacc);
  bp.dkacc = reinterpret_cast<float*>(w + L.dkacc);
  bp.dv_out = dv;
  bp.BH = BH;
  bp.N = N;
  bp.NT = L.fwd.NT;
  bp.KD = L.fwd.KD;
  bp.m = m;
  bp.dv = d_v;
  bp.causal = causal != 0;
  bp.f16_ops = L.fwd.mode == ProjOut::F16X1;
  bp.alpha = static_cast<float>(1.0 / std::sqrt(static_cast<double>(m)));
  bp.limit_ns = limit_ns;
  bp.inject_stall = inject_stall;
  return cuda_status(spa::launch_bwd_tc(bp, stream));
}

// Fused backward, stage 3: dq, dk and dP from dQp and dKp (one tensor-core pass).
int bwd_stage_finish(const void* q, const void* k, const void* P, float* dq, float* dk, float* dP,
                     int B, int H, int N, int d, int m, int d_v, char* w, cudaStream_t stream,
                     unsigned long long limit_ns = kWaitLimitNs, int inject_stall = 0) {
  const BwdLayout L = make_bwd_layout(B, H, N, d, m, d_v, false);
  const int BH = B * H;
  int st;
  spa::BwdFinishParams fp{};
  if ((st = encode_bf16_rows(&fp.qmap, q, d, N, BH)) ||
      (st = encode_bf16_rows(&fp.kmap, k, d, N, BH)) ||
      (st = encode_rows_map(&fp.dqmap, dq, d, N, BH, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4)) ||
      (st = encode_rows_map(&fp.dkmap, dk, d, N, BH, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4)) ||
      (st = device_error_ptr(&fp.err)))
    return st;
  fp.dqacc = reinterpret_cast<const float*>(w + L.dqacc);
  fp.dkacc = reinterpret_cast<const float*>(w + L.dkacc);
  fp.P = static_cast<const __nv_bfloat16*>(P);
  fp.dP = dP;
  fp.B = B;
  fp.H = H;
  fp.N = N;
  fp.NT = L.fwd.NT;
  fp.d = d;
  fp.m = m;
  fp.limit_ns = limit_ns;
  fp.inject_stall = inject_stall;
  return cuda_status(spa::launch_bwd_finish_tc(fp, stream));
}

// The whole fused backward.  lse == NULL: the forward runs once more to
// produce it (into the layout's own lse and scratch output).
int run_backward_fused(const void* q, const void* k, const void* v, const void* P, const float* out,
                       const float* lse, const void* dO, float* dq, float* dk, float* dv,
                       float* dP, int B, int H, int N, int d, int m, int d_v, int causal, char* w,
                       cudaStream_t stream) {
  const BwdLayout L = make_bwd_layout(B, H, N, d, m, d_v, lse == nullptr);
  int st = run_prepare(q, k, P, B, H, N, d, m, SPA_BF16, w, stream, w + L.qb, w + L.kb);
  if (st) return st;
  if (lse == nullptr) {
    float* own = reinterpret_cast<float*>(w + L.lse);
    st = run_apply(v, reinterpret_cast<float*>(w + L.out2), B, H, N, m, d_v, causal, SPA_BF16, w,
                   stream, kWaitLimitNs, 0, own);
    if (st) return st;
    lse = own;
  }
  if ((st = bwd_stage_inputs(out, lse, dO, B, H, N, d, m, d_v, w, stream))) return st;
  if ((st = bwd_stage_kernel(v, dO, dv, B, H, N, d, m, d_v, causal, w, stream))) return st;
  return bwd_stage_finish(q, k, P, dq, dk, dP, B, H, N, d, m, d_v, w, stream);
}

// Checks shared by the staged entry points (fused shapes only).
int check_bwd_staged(int B, int H, int N, int d, int m, int d_v, int dtype, const void* ws,
                     size_t ws_bytes) {
  int st = check_shape(B, H, N, d, m, d_v, dtype);
  if (st) return st;
  if (!bwd_fused_eligible(d, m, d_v, dtype)) return SPA_ERR_UNSUPPORTED;
  if (!ws) return SPA_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(ws) & 255u) return SPA_ERR_ALIGN;
  if (ws_bytes < make_bwd_layout(B, H, N, d, m, d_v, false).total) return SPA_ERR_NOMEM;
  return SPA_OK;
}

// The backward on CUDA cores (fp32 inputs and the shapes the tensor-core
// kernels do not cover): flash-style, nothing N x N stored.  Workspace (from
// the library's pool): Qp, Kp, dQp, dKp in fp32, the row sums <dO_i, O_i>, the
// dP partials, and (without the caller's log-sum-exp) the forward's workspace,
// a scratch output and lse.
int run_backward_simt(const void* q, const void* k, const void* v, const void* P,
                      const float* out, const float* lse, const void* dO, float* dq, float* dk,
                      float* dv, float* dP, int B, int H, int N, int d, int m, int d_v, int causal,
                      int dtype, cudaStream_t s) {
  const size_t BH = static_cast<size_t>(B) * H, rows = BH * N;
  const int chunks = spa::bwd_simt_chunks(B, N);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  const size_t oqp = take(rows * m * 4), okp = take(rows * m * 4), odq = take(rows * m * 4),
               odk = take(rows * m * 4), ods = take(rows * 4),
               opart = take(static_cast<size_t>(H) * chunks * d * m * 4);
  size_t ofw = 0, oout = 0, olse = 0;
  if (!lse) {
    ofw = take(make_layout(B, H, N, m, dtype).total);
    oout = take(rows * d_v * 4);
    olse = take(rows * 4);
  }
  char* w = nullptr;
  if (int e = pool_alloc(reinterpret_cast<void**>(&w), o, s)) return e;
  int st = SPA_OK;
  if (!lse) {  // the forward once more, for its row log-sum-exp
    st = run_prepare(q, k, P, B, H, N, d, m, dtype, w + ofw, s);
    if (!st)
      st = run_apply(v, reinterpret_cast<float*>(w + oout), B, H, N, m, d_v, causal, dtype, w + ofw,
                     s, kWaitLimitNs, 0, reinterpret_cast<float*>(w + olse));
    lse = reinterpret_cast<const float*>(w + olse);
  }
  if (!st) {  // Qp and Kp in fp32
    spa::ProjParams pp{};
    pp.x[0] = q;
    pp.x[1] = k;
    pp.P = P;
    pp.out[0] = w + oqp;
    pp.out[1] = w + okp;
    pp.nx = 2;
    pp.BH = B * H;
    pp.H = H;
    pp.N = N;
    pp.d = d;
    pp.m = m;
    pp.NT = (N + spa::kTileRows - 1) / spa::kTileRows;
    pp.bf16_in = dtype == SPA_BF16;
    pp.mode = ProjOut::F32;
    st = cuda_status(spa::launch_project(pp, s));
  }
  if (!st) {
    spa::BwdSimtParams bp{};
    bp.q = q;
    bp.k = k;
    bp.v = v;
    bp.P = P;
    bp.dO = dO;
    bp.out = out;
    bp.lse = lse;
    bp.dq = dq;
    bp.dk = dk;
    bp.dv_out = dv;
    bp.dP = dP;
    bp.qp = reinterpret_cast<float*>(w + oqp);
    bp.kp = reinterpret_cast<float*>(w + okp);
    bp.dqp = reinterpret_cast<float*>(w + odq);
    bp.dkp = reinterpret_cast<float*>(w + odk);
    bp.dsum = reinterpret_cast<float*>(w + ods);
    bp.part = reinterpret_cast<float*>(w + opart);
    bp.B = B;
    bp.H = H;
    bp.N = N;
    bp.d = d;
    bp.m = m;
    bp.dv = d_v;
    bp.causal = causal != 0;
    bp.bf16 = dtype == SPA_BF16;
    bp.chunks = chunks;
    st = cuda_status(spa::launch_bwd_simt(bp, s));
  }
  const cudaError_t fe = cudaFreeAsync(w, s);
  if (st) return st;
  return cuda_status(fe);
}

// Shared by both backward entry points; lse may be NULL.
int backward_entry(const void* q, const void* k, const void* v, const void* P, const float* out,
                   const float* lse, const void* dO, float* dq, float* dk, float* dv, float* dP,
                   int B, int H, int N, int d, int m, int d_v, int causal, int dtype,
                   void* stream) {
  int st = check_shape(B, H, N, d, m, d_v, dtype);
  if (st == kEmpty) {
    if (!dP) return SPA_ERR_NULL;  // the projection gradient is still defined: zero
    if (H > 0 && d > 0 && m > 0 &&
        cudaMemsetAsync(dP, 0, static_cast<size_t>(H) * d * m * sizeof(float),
                        static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return SPA_ERR_CUDA;
    return SPA_OK;
  }
  if (st) return st;
  if (d > 128) return SPA_ERR_UNSUPPORTED;
  if (!q || !k || !v || !P || !out || !dO || !dq || !dk || !dv || !dP) return SPA_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(P) || !aligned16(dO) ||
      !aligned16(out) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(dP))
    return SPA_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!bwd_fused_eligible(d, m, d_v, dtype))
    return run_backward_simt(q, k, v, P, out, lse, dO, dq, dk, dv, dP, B, H, N, d, m, d_v, causal,
                             dtype, s);
  const size_t bytes = make_bwd_layout(B, H, N, d, m, d_v, lse == nullptr).total;
  void* ws = nullptr;
  if (int e = pool_alloc(&ws, bytes, s)) return e;
  st = run_backward_fused(q, k, v, P, out, lse, dO, dq, dk, dv, dP, B, H, N, d, m, d_v, causal,
                          static_cast<char*>(ws), s);
  const cudaError_t fe = cudaFreeAsync(ws, s);
  if (st) return st;
  return cuda_status(fe);
}

// The Top-k prologue (spa_topk_features), with the wait limit and the
// failure-detection injection of the TMA kernel as parameters.
int topk_features(const void* x, void* y, long long rows, int d, int k, int dtype,
                  cudaStream_t stream, unsigned long long limit_ns = kWaitLimitNs,
                  int inject_stall = 0) {
  if (rows < 0 || d < 0 || k < 0) return SPA_ERR_SHAPE;
  if (dtype != SPA_F32 && dtype != SPA_BF16) return SPA_ERR_DTYPE;
  if (rows == 0) return SPA_OK;
  if (d != 32 && d != 64 && d != 128 && d != 256) return SPA_ERR_UNSUPPORTED;
  if (k < 1 || k > d) return SPA_ERR_SHAPE;
  if (!x || !y) return SPA_ERR_NULL;
  if (!aligned16(x) || !aligned16(y)) return SPA_ERR_ALIGN;
  spa::TopkParams tp{};
  tp.x = x;
  tp.y = y;
  tp.rows = rows;
  tp.d = d;
  tp.k = k;
  tp.bf16 = dtype == SPA_BF16;
  // bf16 rows of 64 or 128 features go through TMA (row coordinates are 32-bit)
  if (tp.bf16 && (d == 64 || d == 128) && rows <= 0x7fffff00LL) {
    int st;
    if ((st = encode_bf16_rows(&tp.xmap, x, d, static_cast<int>(rows), 1)) ||
        (st = encode_bf16_rows(&tp.ymap, y, d, static_cast<int>(rows), 1)) ||
        (st = device_error_ptr(&tp.err)))
      return st;
    tp.use_tma = 1;
    tp.limit_ns = limit_ns;
    tp.inject_stall = inject_stall;
  }
  return cuda_status(spa::launch_topk(tp, stream));
}

}  // namespace

extern "C" {

const char* spa_status_str(int status) {
  switch (status) {
    case SPA_OK: return "SPA_OK";
    case SPA_ERR_NULL: return "SPA_ERR_NULL: a required pointer is NULL";
    case SPA_ERR_SHAPE: return "SPA_ERR_SHAPE: a size is negative or too large";
    case SPA_ERR_DTYPE: return "SPA_ERR_DTYPE: dtype must be SPA_F32 or SPA_BF16";
    case SPA_ERR_ALIGN: return "SPA_ERR_ALIGN: pointers must be 16-byte aligned";
    case SPA_ERR_UNSUPPORTED: return "SPA_ERR_UNSUPPORTED: shape outside the implemented kernels";
    case SPA_ERR_NOMEM: return "SPA_ERR_NOMEM: workspace allocation failed or too small";
    case SPA_ERR_CUDA: return "SPA_ERR_CUDA: a CUDA call failed";
    case SPA_ERR_TIMEOUT: return "SPA_ERR_TIMEOUT: a kernel gave up on a bounded wait";
    default: return "SPA_ERR_UNKNOWN";
  }
}

int spa_version(void) { return 100; }

int spa_project(const void* x, const void* P, float* x_proj, int B, int H, int N, int d, int m,
                int dtype, void* stream) {
  if (B < 0 || H < 0 || N < 0 || d < 0 || m < 0) return SPA_ERR_SHAPE;
  if (dtype != SPA_F32 && dtype != SPA_BF16) return SPA_ERR_DTYPE;
  if (static_cast<long long>(B) * H * N == 0) return SPA_OK;
  if (static_cast<long long>(B) * H > 65535) return SPA_ERR_SHAPE;
  if (d < 1 || d > 256 || m < 1 || m > 128) return SPA_ERR_UNSUPPORTED;
  if (!x || !P || !x_proj) return SPA_ERR_NULL;
  if (!aligned16(x) || !aligned16(P) || !aligned16(x_proj)) return SPA_ERR_ALIGN;
  spa::ProjParams pp{};
  pp.x[0] = x;
  pp.P = P;
  pp.out[0] = x_proj;
  pp.nx = 1;
  pp.BH = B * H;
  pp.H = H;
  pp.N = N;
  pp.d = d;
  pp.m = m;
  pp.NT = (N + spa::kTileRows - 1) / spa::kTileRows;
  pp.bf16_in = dtype == SPA_BF16;
  pp.mode = ProjOut::F32;
  return cuda_status(spa::launch_project(pp, static_cast<cudaStream_t>(stream)));
}

int spa_attention_workspace_size(int B, int H, int N, int d, int m, int d_v, int dtype,
                                 size_t* bytes) {
  if (!bytes) return SPA_ERR_NULL;
  const int st = check_shape(B, H, N, d, m, d_v, dtype);
  if (st == kEmpty) {
    *bytes = 0;
    return SPA_OK;
  }
  if (st) return st;
  *bytes = make_layout(B, H, N, m, dtype).total;
  return SPA_OK;
}

int spa_attention_fwd_ws(const void* q, const void* k, const void* v, const void* P, float* out,
                         int B, int H, int N, int d, int m, int d_v, int causal, int dtype,
                         void* workspace, size_t workspace_bytes, void* stream) {
  int st = check_shape(B, H, N, d, m, d_v, dtype);
  if (st == kEmpty) return SPA_OK;
  if (st) return st;
  if ((st = check_forward_ptrs(q, k, v, P, out))) return st;
  if (!workspace) return SPA_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return SPA_ERR_ALIGN;
  if (workspace_bytes < make_layout(B, H, N, m, dtype).total) return SPA_ERR_NOMEM;
  return run_forward(q, k, v, P, out, B, H, N, d, m, d_v, causal, dtype, workspace,
                     static_cast<cudaStream_t>(stream));
}

int spa_attention_prepare(const void* q, const void* k, const void* P, int B, int H, int N,
                          int d, int m, int d_v, int dtype, void* workspace,
                          size_t workspace_bytes, void* stream) {
  int st = check_shape(B, H, N, d, m, d_v, dtype);
  if (st == kEmpty) return SPA_OK;
  if (st) return st;
  if (!q || !k || !P || !workspace) return SPA_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(P) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return SPA_ERR_ALIGN;
  if (workspace_bytes < make_layout(B, H, N, m, dtype).total) return SPA_ERR_NOMEM;
  return run_prepare(q, k, P, B, H, N, d, m, dtype, workspace, static_cast<cudaStream_t>(stream));
}

int spa_attention_apply(const void* v, float* out, int B, int H, int N, int d, int m, int d_v,
                        int causal, int dtype, const void* workspace, size_t workspace_bytes,
                        void* stream) {
  int st = check_shape(B, H, N, d, m, d_v, dtype);
  if (st == kEmpty) return SPA_OK;
  if (st) return st;
  if (!v || !out || !workspace) return SPA_ERR_NULL;
  if (!aligned16(v) || !aligned16(out) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return SPA_ERR_ALIGN;
  if (workspace_bytes < make_layout(B, H, N, m, dtype).total) return SPA_ERR_NOMEM;
  return run_apply(v, out, B, H, N, m, d_v, causal, dtype, workspace,
                   static_cast<cudaStream_t>(stream));
}

int spa_attention_fwd(const void* q, const void* k, const void* v, const void* P, float* out,
                      int B, int H, int N, int d, int m, int d_v, int causal, int dtype,
                      void* stream) {
  int st = check_shape(B, H, N, d, m, d_v, dtype);
  if (st == kEmpty) return SPA_OK;
  if (st) return st;
  if ((st = check_forward_ptrs(q, k, v, P, out))) return st;
  const size_t bytes = make_layout(B, H, N, m, dtype).total;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* ws = nullptr;
  if (int e = pool_alloc(&ws, bytes, s)) return e;
  st = run_forward(q, k, v, P, out, B, H, N, d, m, d_v, causal, dtype, ws, s);
  const cudaError_t fe = cudaFreeAsync(ws, s);
  if (st) return st;
  return cuda_status(fe);
}

int spa_attention_fwd_host(const void* q, const void* k, const void* v, const void* P,
                           float* out, int B, int H, int N, int d, int m, int d_v, int causal,
                           int dtype, void* stream) {
  int st = check_shape(B, H, N, d, m, d_v, dtype);
  if (st == kEmpty) return SPA_OK;
  if (st) return st;
  if (!q || !k || !v || !P || !out) return SPA_ERR_NULL;
  return host_forward(static_cast<const char*>(q), static_cast<const char*>(k),
                      static_cast<const char*>(v), static_cast<const char*>(P), out, B, H, N, d, m,
                      d_v, causal, dtype, static_cast<cudaStream_t>(stream));
}

int spa_kcache_append(const void* k, const void* P, void* kc, float* kc_mul, int B, int H, int T,
                      int d, int m, int pos, int cap, int dtype, void* stream) {
  if (B < 0 || H < 0 || T < 0 || d < 0 || m < 0 || pos < 0 || cap < 0) return SPA_ERR_SHAPE;
  if (dtype != SPA_F32 && dtype != SPA_BF16) return SPA_ERR_DTYPE;
  if (static_cast<long long>(pos) + T > cap) return SPA_ERR_SHAPE;
  if (static_cast<long long>(B) * H * T == 0) return SPA_OK;
  if (static_cast<long long>(B) * H > 65535) return SPA_ERR_SHAPE;
  if (dtype != SPA_BF16) return SPA_ERR_UNSUPPORTED;
  if (d < 1 || d > 256 || (m != 16 && m != 32 && m != 64 && m != 128)) return SPA_ERR_UNSUPPORTED;
  if (!k || !P || !kc || !kc_mul) return SPA_ERR_NULL;
  if (!aligned16(k) || !aligned16(P) || !aligned16(kc) || !aligned16(kc_mul)) return SPA_ERR_ALIGN;
  // the projection kernels with a row-major fp16 output: rows pos .. pos+T-1
  spa::ProjParams pp{};
  pp.x[0] = k;
  pp.P = P;
  pp.out[0] = kc;
  pp.mul[0] = kc_mul;
  pp.nx = 1;
  pp.BH = B * H;
  pp.H = H;
  pp.N = T;
  pp.d = d;
  pp.m = m;
  pp.NT = (T + spa::kTileRows - 1) / spa::kTileRows;
  pp.qscale = 1.f;
  pp.bf16_in = 1;
  pp.mode = ProjOut::F16ROWS;
  pp.out_rows = cap;
  pp.out_pos = pos;
  pp.use_tc = 1;
  if (spa::project_tc_eligible(pp)) {
    int st;
    if ((st = encode_bf16_rows(&pp.xmap[0], k, d, T, B * H))) return st;
    if ((st = device_error_ptr(&pp.err))) return st;
  }
  return cuda_status(spa::launch_project(pp, static_cast<cudaStream_t>(stream)));
}

int spa_attention_decode(const void* q, const void* P, const void* kc, const float* kc_mul,
                         const void* v, float* out, int B, int H, int L, int d, int m, int d_v,
                         int cap, int dtype, void* stream) {
  if (B < 0 || H < 0 || L < 0 || d < 0 || m < 0 || d_v < 0 || cap < 0) return SPA_ERR_SHAPE;
  if (dtype != SPA_F32 && dtype != SPA_BF16) return SPA_ERR_DTYPE;
  if (static_cast<long long>(B) * H == 0) return SPA_OK;
  if (L < 1 || L > cap) return SPA_ERR_SHAPE;
  if (static_cast<long long>(B) * H > 65535) return SPA_ERR_SHAPE;
  if (dtype != SPA_BF16) return SPA_ERR_UNSUPPORTED;
  if (d < 1 || d > 256 || (m != 16 && m != 32 && m != 64 && m != 128) ||
      (d_v != 64 && d_v != 128))
    return SPA_ERR_UNSUPPORTED;
  if (!q || !P || !kc || !kc_mul || !v || !out) return SPA_ERR_NULL;
  if (!aligned16(q) || !aligned16(P) || !aligned16(kc) || !aligned16(kc_mul) || !aligned16(v) ||
      !aligned16(out))
    return SPA_ERR_ALIGN;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SPA_ERR_CUDA;
  spa::DecodeParams dp{};
  dp.q = static_cast<const __nv_bfloat16*>(q);
  dp.P = static_cast<const __nv_bfloat16*>(P);
  dp.kc = static_cast<const uint16_t*>(kc);
  dp.kc_mul = kc_mul;
  dp.v = static_cast<const __nv_bfloat16*>(v);
  dp.out = out;
  dp.BH = B * H;
  dp.H = H;
  dp.L = L;
  dp.d = d;
  dp.m = m;
  dp.dv = d_v;
  dp.cap = cap;
  dp.qscale = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(m)));
  spa::decode_split(dp.BH, L, sms, &dp.nsplit, &dp.chunk);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t part = static_cast<size_t>(dp.BH) * dp.nsplit * (2 + d_v) * sizeof(float);
  // from the library's own pool, which keeps what it has reserved: a decode loop
  // synchronises every step, and the default pool would hand the scratch back
  // to the driver at each synchronisation and reserve it again on the next call
  cudaMemPool_t pool = nullptr;
  if (host_pool(&pool) != SPA_OK) return SPA_ERR_CUDA;
  if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&dp.part), part, pool, s) != cudaSuccess) {
    cudaGetLastError();
    return SPA_ERR_NOMEM;
  }
  const int st = cuda_status(spa::launch_decode(dp, s));
  const cudaError_t fe = cudaFreeAsync(dp.part, s);
  if (st) return st;
  return fe == cudaSuccess ? SPA_OK : SPA_ERR_CUDA;
}

int spa_topk_features(const void* x, void* y, long long rows, int d, int k, int dtype,
                      void* stream) {
  return topk_features(x, y, rows, d, k, dtype, static_cast<cudaStream_t>(stream));
}

int spa_sfa_attention_fwd(const void* q, const void* k, const void* v, float* out, int B, int H,
                          int N, int d, int d_v, int topk, int causal, int dtype, void* stream) {
  // the forward with P = I_d (m = d): scale 1/sqrt(d) on the sparsified rows
  int st = check_shape(B, H, N, d, d, d_v, dtype);
  if (st == kEmpty) return SPA_OK;
  if (st) return st;
  if (d != 32 && d != 64 && d != 128) return SPA_ERR_UNSUPPORTED;
  if (topk < 1 || topk > d) return SPA_ERR_SHAPE;
  if (!q || !k || !v || !out) return SPA_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return SPA_ERR_ALIGN;
  const size_t es = dtype == SPA_BF16 ? 2 : 4;
  const long long rows = static_cast<long long>(B) * H * N;
  const size_t nq = static_cast<size_t>(rows) * d * es;
  const size_t np = static_cast<size_t>(H) * d * d * es;
  const size_t oq = 0, ok = align256(oq + nq), op = align256(ok + nq), ow = align256(op + np);
  const size_t total = ow + make_layout(B, H, N, d, dtype).total;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* buf = nullptr;
  if (int e = pool_alloc(reinterpret_cast<void**>(&buf), total, s)) return e;
  st = spa_topk_features(q, buf + oq, rows, d, topk, dtype, stream);
  if (!st) st = spa_topk_features(k, buf + ok, rows, d, topk, dtype, stream);
  if (!st) st = cuda_status(spa::launch_identity(buf + op, H, d, dtype == SPA_BF16, s));
  if (!st)
    st = run_forward(buf + oq, buf + ok, v, buf + op, out, B, H, N, d, d, d_v, causal, dtype,
                     buf + ow, s);
  const cudaError_t fe = cudaFreeAsync(buf, s);
  if (st) return st;
  return fe == cudaSuccess ? SPA_OK : SPA_ERR_CUDA;
}

int spa_attention_bwd(const void* q, const void* k, const void* v, const void* P,
                      const float* out, const void* dO, float* dq, float* dk, float* dv,
                      float* dP, int B, int H, int N, int d, int m, int d_v, int causal, int dtype,
                      void* stream) {
  return backward_entry(q, k, v, P, out, nullptr, dO, dq, dk, dv, dP, B, H, N, d, m, d_v, causal,
                        dtype, stream);
}

int spa_attention_bwd_lse(const void* q, const void* k, const void* v, const void* P,
                          const float* out, const float* lse, const void* dO, float* dq, float* dk,
                          float* dv, float* dP, int B, int H, int N, int d, int m, int d_v,
                          int causal, int dtype, void* stream) {
  const int st = check_shape(B, H, N, d, m, d_v, dtype);
  if (st != kEmpty && st) return st;
  if (st != kEmpty && !lse) return SPA_ERR_NULL;
  return backward_entry(q, k, v, P, out, lse, dO, dq, dk, dv, dP, B, H, N, d, m, d_v, causal, dtype,
                        stream);
}

int spa_attention_fwd_lse(const void* q, const void* k, const void* v, const void* P, float* out,
                          float* lse, int B, int H, int N, int d, int m, int d_v, int causal,
                          int dtype, void* stream) {
  int st = check_shape(B, H, N, d, m, d_v, dtype);
  if (st == kEmpty) return SPA_OK;
  if (st) return st;
  if ((st = check_forward_ptrs(q, k, v, P, out))) return st;
  if (!lse) return SPA_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(lse) & 3u) return SPA_ERR_ALIGN;
  const size_t bytes = make_layout(B, H, N, m, dtype).total;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* ws = nullptr;
  if (int e = pool_alloc(&ws, bytes, s)) return e;
  st = run_prepare(q, k, P, B, H, N, d, m, dtype, ws, s);
  if (!st) st = run_apply(v, out, B, H, N, m, d_v, causal, dtype, ws, s, kWaitLimitNs, 0, lse);
  const cudaError_t fe = cudaFreeAsync(ws, s);
  if (st) return st;
  return cuda_status(fe);
}

int spa_attention_bwd_workspace_size(int B, int H, int N, int d, int m, int d_v, int dtype,
                                     size_t* bytes) {
  if (!bytes) return SPA_ERR_NULL;
  const int st = check_shape(B, H, N, d, m, d_v, dtype);
  if (st == kEmpty) {
    *bytes = 0;
    return SPA_OK;
  }
  if (st) return st;
  if (!bwd_fused_eligible(d, m, d_v, dtype)) return SPA_ERR_UNSUPPORTED;
  *bytes = make_bwd_layout(B, H, N, d, m, d_v, false).total;
  return SPA_OK;
}

int spa_attention_bwd_prepare(const void* q, const void* k, const void* P, const float* out,
                              const float* lse, const void* dO, int B, int H, int N, int d, int m,
                              int d_v, int dtype, void* workspace, size_t workspace_bytes,
                              void* stream) {
  int st = check_bwd_staged(B, H, N, d, m, d_v, dtype, workspace, workspace_bytes);
  if (st == kEmpty) return SPA_OK;
  if (st) return st;
  if (!q || !k || !P || !out || !lse || !dO) return SPA_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(P) || !aligned16(out) || !aligned16(dO))
    return SPA_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(workspace);
  const BwdLayout L = make_bwd_layout(B, H, N, d, m, d_v, false);
  if ((st = run_prepare(q, k, P, B, H, N, d, m, SPA_BF16, w, s, w + L.qb, w + L.kb))) return st;
  return bwd_stage_inputs(out, lse, dO, B, H, N, d, m, d_v, w, s);
}

int spa_attention_bwd_apply(const void* v, const void* dO, float* dv, int B, int H, int N, int d,
                            int m, int d_v, int causal, int dtype, void* workspace,
                            size_t workspace_bytes, void* stream) {
  int st = check_bwd_staged(B, H, N, d, m, d_v, dtype, workspace, workspace_bytes);
  if (st == kEmpty) return SPA_OK;
  if (st) return st;
  if (!v || !dO || !dv) return SPA_ERR_NULL;
  if (!aligned16(v) || !aligned16(dO) || !aligned16(dv)) return SPA_ERR_ALIGN;
  return bwd_stage_kernel(v, dO, dv, B, H, N, d, m, d_v, causal, static_cast<char*>(workspace),
                          static_cast<cudaStream_t>(stream));
}

int spa_attention_bwd_finish(const void* q, const void* k, const void* P, float* dq, float* dk,
                             float* dP, int B, int H, int N, int d, int m, int d_v, int dtype,
                             void* workspace, size_t workspace_bytes, void* stream) {
  int st = check_bwd_staged(B, H, N, d, m, d_v, dtype, workspace, workspace_bytes);
  if (st == kEmpty) {
    if (!dP) return SPA_ERR_NULL;
    if (H > 0 && d > 0 && m > 0 &&
        cudaMemsetAsync(dP, 0, static_cast<size_t>(H) * d * m * sizeof(float),
                        static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return SPA_ERR_CUDA;
    return SPA_OK;
  }
  if (st) return st;
  if (!q || !k || !P || !dq || !dk || !dP) return SPA_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(P) || !aligned16(dq) || !aligned16(dk) ||
      !aligned16(dP))
    return SPA_ERR_ALIGN;
  return bwd_stage_finish(q, k, P, dq, dk, dP, B, H, N, d, m, d_v, static_cast<char*>(workspace),
                          static_cast<cudaStream_t>(stream));
}

int spa_host_pool_trim(void) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_host_pool_mu);
  if (g_host_pool[dev] && cudaMemPoolTrimTo(g_host_pool[dev], 0) != cudaSuccess) return SPA_ERR_CUDA;
  return SPA_OK;
}

int spa_selftest_wait_timeout(int limit_ms) {
  if (limit_ms <= 0 || limit_ms > 2000) return SPA_ERR_SHAPE;
  constexpr int B = 1, H = 1, N = 256, d = 64, m = 32, dv = 64;
  const size_t nq = static_cast<size_t>(N) * d * 2, nv = static_cast<size_t>(N) * dv * 2;
  const size_t np = static_cast<size_t>(d) * m * 2, no = static_cast<size_t>(N) * dv * 4;
  const size_t oq = 0, ok = align256(oq + nq), ov = align256(ok + nq), op = align256(ov + nv),
               oo = align256(op + np), ow = align256(oo + no);
  const size_t total = ow + make_layout(B, H, N, m, SPA_BF16).total;
  int* err = nullptr;
  int st = device_error_ptr(&err);
  if (st) return st;
  char* buf = nullptr;
  if (cudaMalloc(reinterpret_cast<void**>(&buf), total) != cudaSuccess) {
    cudaGetLastError();
    return SPA_ERR_NOMEM;
  }
  st = cuda_status(cudaMemset(buf, 0, total));  // zero inputs: every score is 0
  if (!st) st = run_prepare(buf + oq, buf + ok, buf + op, B, H, N, d, m, SPA_BF16, buf + ow, nullptr);
  if (!st)
    st = run_apply(buf + ov, reinterpret_cast<float*>(buf + oo), B, H, N, m, dv, 0, SPA_BF16,
                   buf + ow, nullptr, static_cast<unsigned long long>(limit_ms) * 1000000ull, 1);
  if (!st) st = cuda_status(cudaDeviceSynchronize());
  int word = 0;
  if (!st) st = cuda_status(cudaMemcpy(&word, err, sizeof word, cudaMemcpyDeviceToHost));
  const int zero = 0;
  if (!st) st = cuda_status(cudaMemcpy(err, &zero, sizeof zero, cudaMemcpyHostToDevice));
  cudaFree(buf);
  if (st) return st;
  return word ? SPA_ERR_TIMEOUT : SPA_OK;
}

int spa_selftest_proj_wait_timeout(int limit_ms, int m) {
  if (limit_ms <= 0 || limit_ms > 2000) return SPA_ERR_SHAPE;
  if (m != 32 && m != 64) return SPA_ERR_UNSUPPORTED;
  // m = 32 runs the per-CTA projection kernel, m = 64 the warp-specialised
  // one; 512 tiles, so each CTA of either takes one to four of them
  constexpr int B = 1, H = 8, N = 4096, d = 64;
  const size_t nq = static_cast<size_t>(B) * H * N * d * 2, np = static_cast<size_t>(H) * d * m * 2;
  const size_t oq = 0, ok = align256(oq + nq), op = align256(ok + nq), ow = align256(op + np);
  const size_t total = ow + make_layout(B, H, N, m, SPA_BF16).total;
  int* err = nullptr;
  int st = device_error_ptr(&err);
  if (st) return st;
  char* buf = nullptr;
  if (cudaMalloc(reinterpret_cast<void**>(&buf), total) != cudaSuccess) {
    cudaGetLastError();
    return SPA_ERR_NOMEM;
  }
  st = cuda_status(cudaMemset(buf, 0, total));  // zero inputs
  if (!st)
    st = run_prepare(buf + oq, buf + ok, buf + op, B, H, N, d, m, SPA_BF16, buf + ow, nullptr,
                     nullptr, nullptr, static_cast<unsigned long long>(limit_ms) * 1000000ull, 1);
  if (!st) st = cuda_status(cudaDeviceSynchronize());
  int word = 0;
  if (!st) st = cuda_status(cudaMemcpy(&word, err, sizeof word, cudaMemcpyDeviceToHost));
  const int zero = 0;
  if (!st) st = cuda_status(cudaMemcpy(err, &zero, sizeof zero, cudaMemcpyHostToDevice));
  cudaFree(buf);
  if (st) return st;
  return word ? SPA_ERR_TIMEOUT : SPA_OK;
}

int spa_selftest_copy_wait_timeout(int limit_ms, int kernel) {
  if (limit_ms <= 0 || limit_ms > 2000) return SPA_ERR_SHAPE;
  if (kernel < 0 || kernel > 2) return SPA_ERR_UNSUPPORTED;
  // 8 heads of 4096 rows (d = 64, m = 32, d_v = 128): 256 row blocks for the
  // statistics and the Top-k kernels, 512 tiles for the finish
  constexpr int B = 1, H = 8, N = 4096, d = 64, m = 32, dv = 128, topk_d = 128, topk_k = 16;
  const size_t rows = static_cast<size_t>(B) * H * N;
  const BwdLayout L = make_bwd_layout(B, H, N, d, m, dv, false);
  const size_t nx = rows * d * 2, np = static_cast<size_t>(H) * d * m * 2;
  const size_t ndo = rows * dv * 2, nout = rows * dv * 4, nlse = rows * 4, ng = rows * d * 4;
  const size_t ndp = static_cast<size_t>(H) * d * m * 4, nt = rows * topk_d * 2;
  const size_t oq = 0, ok = align256(oq + nx), op = align256(ok + nx), odo = align256(op + np),
               oo = align256(odo + ndo), ol = align256(oo + nout), odq = align256(ol + nlse),
               odk = align256(odq + ng), odp = align256(odk + ng), ox = align256(odp + ndp),
               oy = align256(ox + nt), ow = align256(oy + nt);
  const size_t total = ow + L.total;
  int* err = nullptr;
  int st = device_error_ptr(&err);
  if (st) return st;
  char* buf = nullptr;
  if (cudaMalloc(reinterpret_cast<void**>(&buf), total) != cudaSuccess) {
    cudaGetLastError();
    return SPA_ERR_NOMEM;
  }
  st = cuda_status(cudaMemset(buf, 0, total));  // zero inputs, statistics and accumulators
  const unsigned long long lim = static_cast<unsigned long long>(limit_ms) * 1000000ull;
  char* w = buf + ow;
  if (!st && kernel == 0)
    st = bwd_stage_inputs(reinterpret_cast<const float*>(buf + oo),
                          reinterpret_cast<const float*>(buf + ol), buf + odo, B, H, N, d, m, dv, w,
                          nullptr, lim, 1);
  if (!st && kernel == 1)
    st = bwd_stage_finish(buf + oq, buf + ok, buf + op, reinterpret_cast<float*>(buf + odq),
                          reinterpret_cast<float*>(buf + odk), reinterpret_cast<float*>(buf + odp),
                          B, H, N, d, m, dv, w, nullptr, lim, 1);
  if (!st && kernel == 2)
    st = topk_features(buf + ox, buf + oy, static_cast<long long>(rows), topk_d, topk_k, SPA_BF16,
                       nullptr, lim, 1);
  if (!st) st = cuda_status(cudaDeviceSynchronize());
  int word = 0;
  if (!st) st = cuda_status(cudaMemcpy(&word, err, sizeof word, cudaMemcpyDeviceToHost));
  const int zero = 0;
  if (!st) st = cuda_status(cudaMemcpy(err, &zero, sizeof zero, cudaMemcpyHostToDevice));
  cudaFree(buf);
  if (st) return st;
  return word ? SPA_ERR_TIMEOUT : SPA_OK;
}

int spa_selftest_bwd_wait_timeout(int limit_ms) {
  if (limit_ms <= 0 || limit_ms > 2000) return SPA_ERR_SHAPE;
  constexpr int B = 1, H = 1, N = 256, d = 64, m = 32, dv = 64;
  const size_t nq = static_cast<size_t>(N) * d * 2, nv = static_cast<size_t>(N) * dv * 2;
  const size_t np = static_cast<size_t>(d) * m * 2, no = static_cast<size_t>(N) * dv * 4;
  const size_t nl = static_cast<size_t>(N) * 4;
  const size_t oq = 0, ok = align256(oq + nq), ov = align256(ok + nq), op = align256(ov + nv),
               odo = align256(op + np), oo = align256(odo + nv), ol = align256(oo + no),
               odv = align256(ol + nl), ow = align256(odv + no);
  const BwdLayout L = make_bwd_layout(B, H, N, d, m, dv, false);
  const size_t total = ow + L.total;
  int* err = nullptr;
  int st = device_error_ptr(&err);
  if (st) return st;
  char* buf = nullptr;
  if (cudaMalloc(reinterpret_cast<void**>(&buf), total) != cudaSuccess) {
    cudaGetLastError();
    return SPA_ERR_NOMEM;
  }
  // zero inputs and log-sum-exp: every value the kernel computes is finite
  st = cuda_status(cudaMemset(buf, 0, total));
  char* w = buf + ow;
  if (!st)
    st = run_prepare(buf + oq, buf + ok, buf + op, B, H, N, d, m, SPA_BF16, w, nullptr, w + L.qb,
                     w + L.kb);
  if (!st)
    st = bwd_stage_inputs(reinterpret_cast<const float*>(buf + oo),
                          reinterpret_cast<const float*>(buf + ol), buf + odo, B, H, N, d, m, dv, w,
                          nullptr);
  if (!st)
    st = bwd_stage_kernel(buf + ov, buf + odo, reinterpret_cast<float*>(buf + odv), B, H, N, d, m,
                          dv, 1, w, nullptr, static_cast<unsigned long long>(limit_ms) * 1000000ull,
                          1);
  if (!st) st = cuda_status(cudaDeviceSynchronize());
  int word = 0;
  if (!st) st = cuda_status(cudaMemcpy(&word, err, sizeof word, cudaMemcpyDeviceToHost));
  const int zero = 0;
  if (!st) st = cuda_status(cudaMemcpy(err, &zero, sizeof zero, cudaMemcpyHostToDevice));
  cudaFree(buf);
  if (st) return st;
  return word ? SPA_ERR_TIMEOUT : SPA_OK;
}

int spa_device_error(int* code) {
  if (!code) return SPA_ERR_NULL;
  int* p = nullptr;
  int st = device_error_ptr(&p);
  if (st) return st;
  if (cudaDeviceSynchronize() != cudaSuccess) return SPA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, p, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return SPA_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpy(p, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return SPA_ERR_CUDA;
  *code = v ? SPA_ERR_TIMEOUT : SPA_OK;
  return SPA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free forward.  Some callers cannot allocate device memory while
// they run: code that executes inside a framework that owns all device memory
// and forbids cudaMalloc (or is itself inside an allocator callback), real-time
// loops that must not touch the driver's allocator, or processes whose memory
// budget is fixed up front.  For them the forward can use a scratch buffer that
// the library carries as a file-scope device array, sized once at compile time.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB per device

// Scratch for the score-operand tiles / projections of spa_attention_fwd_noalloc.
// In host code this symbol is only a stand-in: its device address comes from
// cudaGetSymbolAddress, taken per device below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

void* g_noalloc_ptr[kMaxDevices] = {};
std::mutex g_noalloc_mu;

// Once per device, with that device current: the device address of the array.
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SPA_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return SPA_OK;
}

}  // namespace

extern "C" int spa_attention_fwd_noalloc(const void* q, const void* k, const void* v,
                                         const void* P, float* out, int B, int H, int N, int d,
                                         int m, int d_v, int causal, int dtype, void* stream) {
  int st = check_shape(B, H, N, d, m, d_v, dtype);
  if (st == kEmpty) return SPA_OK;
  if (st) return st;
  if ((st = check_forward_ptrs(q, k, v, P, out))) return st;
  if (make_layout(B, H, N, m, dtype).total > kNoAllocScratchBytes) return SPA_ERR_NOMEM;
  void* scratch = nullptr;
  if ((st = noalloc_scratch(&scratch))) return st;
  // Every scratch byte the attention stage reads is written first by this
  // call's projection stage, so nothing has to be cleared between calls.
  return run_forward(q, k, v, P, out, B, H, N, d, m, d_v, causal, dtype, scratch,
                     static_cast<cudaStream_t>(stream));
}
