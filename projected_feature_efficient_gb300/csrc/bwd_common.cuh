// bwd_common.cuh -- device helpers shared by the two backward kernels
// (bwd_ws.cu, bwd_finish.cu): the bulk fp32 reduce-add into global memory and
// the bf16 hi | lo split of the gradients.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

#include "ptx.cuh"

namespace spa {

// Tile layout of the fp32 gradient accumulators dQp and dKp the fused kernel
// writes and the finish kernel reads: per 128-row tile, m / W slabs of
// 128 rows x W columns (W = dq_slab_cols(m)), one after the other; within a
// slab, 16-byte chunk q of row e sits at chunk q ^ dq_slab_swizzle(e, W)
// (which spreads a warp's row-per-thread accesses over the banks).
__host__ __device__ constexpr int dq_slab_cols(int m) { return m > 32 ? 16 : m; }
__host__ __device__ constexpr uint32_t dq_slab_swizzle(int e, int W) {
  return static_cast<uint32_t>((e * W / 32) & (W / 4 - 1));
}

// Bulk reduce-add shared -> global (fp32 add, element-wise), tracked by bulk groups.
__device__ __forceinline__ void bulk_reduce_add_f32(float* gdst, uint32_t ssrc, uint32_t bytes) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(
                   gdst),
               "r"(ssrc), "r"(bytes)
               : "memory");
}

// v = hi + lo with hi = bf16(v), lo = bf16(v - hi): two values at a time as
// bf16 pairs (16 significant bits of each value)
__device__ __forceinline__ void split_pair(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat16 ha = __float2bfloat16_rn(a), hb = __float2bfloat16_rn(b);
  hi = static_cast<uint32_t>(__bfloat16_as_ushort(ha)) |
       (static_cast<uint32_t>(__bfloat16_as_ushort(hb)) << 16);
  lo = ptx::pack_bf16x2(a - __bfloat162float(ha), b - __bfloat162float(hb));
}

}  // namespace spa
