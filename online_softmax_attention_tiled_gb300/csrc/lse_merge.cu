// lse_merge.cu -- merge of split partials by their log-sum-exp.
//
// For each row r with S partials (normalised output o_c, lse_c):
//   L = max_c lse_c, w_c = exp(lse_c - L), W = sum_c w_c,
//   lse = L + ln W, o = (sum_c w_c o_c) / W.
// This is the (m, l) merge of the interview lesson (Step 1) written for
// normalised partials (Step 2's rule): a partial's (m, l) is (lse_c, 1).
// A partial with lse_c = -inf has weight exactly zero; if every partial is
// -inf the row is +0.0 with lse -inf (0 is the reference, never -inf - -inf).
// One warp per row; 128-bit loads of the partial outputs when d % 4 == 0.
#include "oa_internal.h"

namespace oa {
namespace {

constexpr int kWarpsPerBlock = 8;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

template <bool VEC, bool OUT_BF16>
__global__ void __launch_bounds__(kWarpsPerBlock * 32) lse_merge_kernel(const float* __restrict__ part_o,
                                                                         const float* __restrict__ part_lse,
                                                                         int S, int64_t R, int d, void* o,
                                                                         float* __restrict__ lse) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  if (row >= R) return;

  float L = -INFINITY;
  for (int c = lane; c < S; c += 32) L = fmaxf(L, part_lse[(int64_t)c * R + row]);
  L = warp_max(L);
  float W = 0.f;
  if (L != -INFINITY)
    for (int c = lane; c < S; c += 32) W += expf(part_lse[(int64_t)c * R + row] - L);
  W = warp_sum(W);

  if (lse != nullptr && lane == 0) lse[row] = (L == -INFINITY) ? -INFINITY : L + logf(W);
  if (d == 0) return;
  const float inv_w = (L == -INFINITY) ? 0.f : 1.f / W;

  if constexpr (VEC) {
    for (int e = lane * 4; e < d; e += 128) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      if (L != -INFINITY) {
        for (int c = 0; c < S; ++c) {
          const float lc = __ldg(part_lse + (int64_t)c * R + row);
          if (lc == -INFINITY) continue;
          const float w = expf(lc - L);
          const float4 pv = __ldg(reinterpret_cast<const float4*>(part_o + ((int64_t)c * R + row) * d + e));
          acc.x = fmaf(w, pv.x, acc.x);
          acc.y = fmaf(w, pv.y, acc.y);
          acc.z = fmaf(w, pv.z, acc.z);
          acc.w = fmaf(w, pv.w, acc.w);
        }
      }
      acc.x *= inv_w, acc.y *= inv_w, acc.z *= inv_w, acc.w *= inv_w;
      if constexpr (OUT_BF16) {
        uint2 pk;
        pk.x = pack_bf16x2(acc.x, acc.y);
        pk.y = pack_bf16x2(acc.z, acc.w);
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(o) + row * d + e) = pk;
      } else {
        *reinterpret_cast<float4*>(static_cast<float*>(o) + row * d + e) = acc;
      }
    }
  } else {
    for (int e = lane; e < d; e += 32) {
      float acc = 0.f;
      if (L != -INFINITY) {
        for (int c = 0; c < S; ++c) {
          const float lc = __ldg(part_lse + (int64_t)c * R + row);
          if (lc == -INFINITY) continue;
          acc = fmaf(expf(lc - L), __ldg(part_o + ((int64_t)c * R + row) * d + e), acc);
        }
      }
      acc *= inv_w;
      if constexpr (OUT_BF16)
        static_cast<__nv_bfloat16*>(o)[row * d + e] = __float2bfloat16_rn(acc);
      else
        static_cast<float*>(o)[row * d + e] = acc;
    }
  }
}

}  // namespace

cudaError_t launch_lse_merge(const float* part_o, const float* part_lse, int S, int64_t R, int d, void* o,
                             bool o_bf16, float* lse, cudaStream_t s) {
  const bool vec = d > 0 && d % 4 == 0 && reinterpret_cast<uintptr_t>(part_o) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(o) % (o_bf16 ? 8 : 16) == 0;
  const dim3 grid((unsigned)((R + kWarpsPerBlock - 1) / kWarpsPerBlock));
  const dim3 block(kWarpsPerBlock * 32);
  if (vec) {
    if (o_bf16)
      lse_merge_kernel<true, true><<<grid, block, 0, s>>>(part_o, part_lse, S, R, d, o, lse);
    else
      lse_merge_kernel<true, false><<<grid, block, 0, s>>>(part_o, part_lse, S, R, d, o, lse);
  } else {
    if (o_bf16)
      lse_merge_kernel<false, true><<<grid, block, 0, s>>>(part_o, part_lse, S, R, d, o, lse);
    else
      lse_merge_kernel<false, false><<<grid, block, 0, s>>>(part_o, part_lse, S, R, d, o, lse);
  }
  return cudaGetLastError();
}

}  // namespace oa
