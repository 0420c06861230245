// Log-sum-exp merge of split-KV partials (workspace.py page, bullet 14: the
// decode_o_part / decode_ml_part buffers).  One warp per (b, query head):
//   M = max over non-empty splits of m_s,  w_s = l_s * exp(m_s - M),
//   out = sum_s w_s o_s / sum_s w_s,  lse = M + ln(sum_s w_s).
#include "kernels.cuh"

namespace pkv {

namespace {

constexpr int kMergeWarps = 4;

template <int D>
__global__ void __launch_bounds__(kMergeWarps * 32)
    merge_kernel(pkv_workspace ws, int batch, int S, int flags) {
  const int lane = threadIdx.x & 31;
  const long long wg = (long long)blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
  const int Hq = ws.n_q_heads;
  if (wg >= (long long)batch * Hq) return;
  const float *ml = ws.ml_part + wg * S * 2;
  const float *op = ws.o_part + wg * S * D;
  constexpr int NV = D / 4;  // float4 vectors per row
  static_assert(NV <= 32, "one float4 per lane");

  float M = -INFINITY;
  for (int s = lane; s < S; s += 32)
    if (ml[2 * s + 1] > 0.f) M = fmaxf(M, ml[2 * s]);
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, d));

  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < S; ++s) {
      const float l = ml[2 * s + 1];
      if (l > 0.f) {
        const float w = l * expf(ml[2 * s] - M);
        den += w;
        if (lane < NV) {
          const float4 o = reinterpret_cast<const float4 *>(op + (long long)s * D)[lane];
          acc.x = fmaf(w, o.x, acc.x);
          acc.y = fmaf(w, o.y, acc.y);
          acc.z = fmaf(w, o.z, acc.z);
          acc.w = fmaf(w, o.w, acc.w);
        }
      }
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  if (lane < NV) {
    const float4 r = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    if (flags & PKV_FLAG_OUT_F32) {
      reinterpret_cast<float4 *>(static_cast<float *>(ws.out) + wg * D)[lane] = r;
    } else {
      uint2 pk;
      pk.x = f32_to_bf16_bits(r.x) | (f32_to_bf16_bits(r.y) << 16);
      pk.y = f32_to_bf16_bits(r.z) | (f32_to_bf16_bits(r.w) << 16);
      reinterpret_cast<uint2 *>(static_cast<uint16_t *>(ws.out) + wg * D)[lane] = pk;
    }
  }
  if (lane == 0 && (flags & PKV_FLAG_WRITE_LSE) && ws.lse)
    ws.lse[wg] = den > 0.f ? M + logf(den) : -INFINITY;
}

}  // namespace

cudaError_t launch_merge(const pkv_workspace &ws, int batch, int num_splits, int flags,
                         cudaStream_t st) {
  const long long pairs = (long long)batch * ws.n_q_heads;
  const int grid = (int)((pairs + kMergeWarps - 1) / kMergeWarps);
  if (grid <= 0) return cudaSuccess;
  if (ws.head_dim == 128)
    merge_kernel<128><<<grid, kMergeWarps * 32, 0, st>>>(ws, batch, num_splits, flags);
  else if (ws.head_dim == 64)
    merge_kernel<64><<<grid, kMergeWarps * 32, 0, st>>>(ws, batch, num_splits, flags);
  else
    return cudaErrorNotSupported;
  return cudaGetLastError();
}

}  // namespace pkv
