// Log-sum-exp merge of one (request, query head) row's split partials by one
// warp (workspace.py page, bullet 14: decode_o_part / decode_ml_part):
//   M = max over non-empty splits of m_s,  w_s = l_s * exp(m_s - M),
//   out = sum_s w_s o_s / sum_s w_s,  lse = M + ln(sum_s w_s).
// Splits come in chunks of 32, lane s holding split s's (m, l); the chunk's
// first eight partial rows are loaded together with the (m, l) pairs and the
// rest eight at a time, every load of a group in flight at once (they may
// come from other CTAs, so L2 loads).  A row of more than 32 splits rebases
// the earlier chunks' sums onto the running maximum.
#pragma once

#include "common.cuh"

namespace pkv {

template <int D>
__device__ __forceinline__ void merge_row(const float *ml, const float *op, int n, int lane,
                                          float &M_out, float &den_out, float4 &acc_out) {
  constexpr int NV = D / 4;  // float4 vectors per row
  constexpr int GS = 8;      // partial rows per group of loads
  static_assert(NV <= 32, "one float4 per lane");
  const float2 *ml2 = reinterpret_cast<const float2 *>(ml);
  float M = -INFINITY, den = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < n; s0 += 32) {
    const int m = min(32, n - s0);
    float2 v = make_float2(-INFINITY, 0.f);
    if (lane < m) v = __ldcg(ml2 + s0 + lane);
    float4 oj[GS];
#pragma unroll
    for (int t = 0; t < GS; ++t)
      oj[t] = (t < m && lane < NV)
                  ? __ldcg(reinterpret_cast<const float4 *>(op + (long long)(s0 + t) * D) + lane)
                  : make_float4(0.f, 0.f, 0.f, 0.f);
    float mc = v.y > 0.f ? v.x : -INFINITY;
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, d));
    const float Mn = fmaxf(M, mc);
    if (Mn == -INFINITY) continue;  // no non-empty split yet
    if (M != -INFINITY && Mn != M) {
      const float sc = expf(M - Mn);
      den *= sc;
      acc = make_float4(acc.x * sc, acc.y * sc, acc.z * sc, acc.w * sc);
    }
    M = Mn;
    const float w = v.y > 0.f ? v.y * expf(v.x - M) : 0.f;
    den += w;
    for (int j = 0; j < m; j += GS) {
      if (j > 0) {
#pragma unroll
        for (int t = 0; t < GS; ++t)
          oj[t] = (j + t < m && lane < NV)
                      ? __ldcg(reinterpret_cast<const float4 *>(op + (long long)(s0 + j + t) * D) +
                               lane)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int t = 0; t < GS; ++t) {
        const float wj = __shfl_sync(0xffffffffu, w, (j + t) & 31);
        if (j + t < m && wj > 0.f) {
          acc.x = fmaf(wj, oj[t].x, acc.x);
          acc.y = fmaf(wj, oj[t].y, acc.y);
          acc.z = fmaf(wj, oj[t].z, acc.z);
          acc.w = fmaf(wj, oj[t].w, acc.w);
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

// Merge of the n split partials of NH query-head rows (row0 + j * rstep,
// j < NH) by one warp, with all of a group of partial-row loads in flight:
// lane s holds split s's weight for every row, and GS splits x NH rows of
// float4 loads are issued before any is used (the first group together with
// the weights' loads).
template <int D, int NH>
__device__ __forceinline__ void merge_rows_batched(const pkv_workspace &ws, long long row0,
                                                   long long rstep, int S, int n, int flags,
                                                   int lane) {
  constexpr int NV = D / 4;
  float M[NH], den[NH];
  float4 acc[NH];
#pragma unroll
  for (int j = 0; j < NH; ++j) {
    M[j] = -INFINITY;
    den[j] = 0.f;
    acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  constexpr int GS = NH >= 4 ? 4 : (NH == 1 ? 16 : 8);  // splits per group of row loads
  auto load_rows = [&](float4 (&o)[GS][NH], int s, int m) {  // splits s .. s + GS - 1 (< m)
#pragma unroll
    for (int t = 0; t < GS; ++t)
#pragma unroll
      for (int j = 0; j < NH; ++j)
        o[t][j] = (t < m && lane < NV)
                      ? __ldcg(reinterpret_cast<const float4 *>(
                                   ws.o_part + ((row0 + j * rstep) * S + s + t) * D) + lane)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
  };
  for (int s0 = 0; s0 < n; s0 += 32) {
    // (m, l) of split s0 + lane for every row, with the first GS splits' rows
    // (independent of the weights) already in flight
    float2 ml[NH];
#pragma unroll
    for (int j = 0; j < NH; ++j)
      ml[j] = s0 + lane < n
                  ? __ldcg(reinterpret_cast<const float2 *>(ws.ml_part + (row0 + j * rstep) * S * 2) + s0 + lane)
                  : make_float2(-INFINITY, 0.f);
    const int m = min(32, n - s0);
    float4 o[GS][NH];
    load_rows(o, s0, m);
    float w[NH];
#pragma unroll
    for (int j = 0; j < NH; ++j) {
      float mx = ml[j].y > 0.f ? ml[j].x : -INFINITY;
#pragma unroll
      for (int d = 16; d >= 1; d >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, d));
      const float Mn = fmaxf(M[j], mx);
      // rescale what was accumulated against the old maximum
      const float r = M[j] == -INFINITY ? 0.f : expf(M[j] - Mn);
      den[j] *= r;
      acc[j].x *= r;
      acc[j].y *= r;
      acc[j].z *= r;
      acc[j].w *= r;
      M[j] = Mn;
      w[j] = (ml[j].y > 0.f && Mn != -INFINITY) ? ml[j].y * expf(ml[j].x - Mn) : 0.f;
      float ws_ = w[j];
#pragma unroll
      for (int d = 16; d >= 1; d >>= 1) ws_ += __shfl_xor_sync(0xffffffffu, ws_, d);
      den[j] += ws_;
    }
    for (int t0 = 0; t0 < m; t0 += GS) {
      if (t0 > 0) load_rows(o, s0 + t0, m - t0);
#pragma unroll
      for (int t = 0; t < GS; ++t)
#pragma unroll
        for (int j = 0; j < NH; ++j) {
          const float wt = __shfl_sync(0xffffffffu, w[j], (t0 + t) & 31);
          if (t0 + t < m && wt > 0.f) {
            acc[j].x = fmaf(wt, o[t][j].x, acc[j].x);
            acc[j].y = fmaf(wt, o[t][j].y, acc[j].y);
            acc[j].z = fmaf(wt, o[t][j].z, acc[j].z);
            acc[j].w = fmaf(wt, o[t][j].w, acc[j].w);
          }
        }
    }
  }
#pragma unroll
  for (int j = 0; j < NH; ++j) merge_store<D>(ws, row0 + j * rstep, flags, lane, M[j], den[j], acc[j]);
}

}  // namespace pkv
