// Log-sum-exp merge of one (request, query head) row's split partials by one
// warp (workspace.py page, bullet 14: decode_o_part / decode_ml_part):
//   M = max over non-empty splits of m_s,  w_s = l_s * exp(m_s - M),
//   out = sum_s w_s o_s / sum_s w_s,  lse = M + ln(sum_s w_s).
// Lane s holds split s's (m, l); the partial rows are then read four at a
// time with independent L2 loads (they may come from other CTAs).
#pragma once

#include "common.cuh"

namespace pkv {

template <int D>
__device__ __forceinline__ void merge_row(const float *ml, const float *op, int n, int lane,
                                          float &M_out, float &den_out, float4 &acc_out) {
  constexpr int NV = D / 4;  // float4 vectors per row
  static_assert(NV <= 32, "one float4 per lane");
  const float2 *ml2 = reinterpret_cast<const float2 *>(ml);
  float M = -INFINITY;
  for (int s = lane; s < n; s += 32) {
    const float2 v = __ldcg(ml2 + s);
    if (v.y > 0.f) M = fmaxf(M, v.x);
  }
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, d));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
  if (M != -INFINITY) {
    for (int s0 = 0; s0 < n; s0 += 32) {
      float w = 0.f;
      if (s0 + lane < n) {
        const float2 v = __ldcg(ml2 + s0 + lane);
        w = v.y > 0.f ? v.y * expf(v.x - M) : 0.f;
      }
      den += w;
      const int m = min(32, n - s0);
      for (int j = 0; j < m; j += 4) {
        float wj[4];
        float4 oj[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) wj[t] = __shfl_sync(0xffffffffu, w, (j + t) & 31);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          oj[t] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (j + t < m && lane < NV)
            oj[t] = __ldcg(reinterpret_cast<const float4 *>(op + (long long)(s0 + j + t) * D) + lane);
        }
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          if (j + t < m && wj[t] > 0.f) {
            acc.x = fmaf(wj[t], oj[t].x, acc.x);
            acc.y = fmaf(wj[t], oj[t].y, acc.y);
            acc.z = fmaf(wj[t], oj[t].z, acc.z);
            acc.w = fmaf(wj[t], oj[t].w, acc.w);
          }
        }
      }
    }
  }
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) den += __shfl_xor_sync(0xffffffffu, den, d);
  M_out = M;
  den_out = den;
  acc_out = acc;
}

// Write one merged row: out (bf16 or fp32 by flag) and, if asked, lse.
template <int D>
__device__ __forceinline__ void merge_store(const pkv_workspace &ws, long long row, int flags,
                                            int lane, float M, float den, float4 acc) {
  constexpr int NV = D / 4;
  const float inv = den > 0.f ? 1.f / den : 0.f;
  if (lane < NV) {
    const float4 r = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    if (flags & PKV_FLAG_OUT_F32) {
      reinterpret_cast<float4 *>(static_cast<float *>(ws.out) + row * D)[lane] = r;
    } else {
      uint2 pk;
      pk.x = f32_to_bf16_bits(r.x) | (f32_to_bf16_bits(r.y) << 16);
      pk.y = f32_to_bf16_bits(r.z) | (f32_to_bf16_bits(r.w) << 16);
      reinterpret_cast<uint2 *>(static_cast<uint16_t *>(ws.out) + row * D)[lane] = pk;
    }
  }
  if (lane == 0 && (flags & PKV_FLAG_WRITE_LSE) && ws.lse)
    ws.lse[row] = den > 0.f ? M + logf(den) : -INFINITY;
}

}  // namespace pkv
