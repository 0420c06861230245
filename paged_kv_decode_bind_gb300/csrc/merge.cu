// Log-sum-exp merge of split-KV partials (workspace.py page, bullet 14: the
// decode_o_part / decode_ml_part buffers).  One warp per (b, query head):
//   M = max over non-empty splits of m_s,  w_s = l_s * exp(m_s - M),
//   out = sum_s w_s o_s / sum_s w_s,  lse = M + ln(sum_s w_s).
#include "decode_plan.cuh"
#include "kernels.cuh"
#include "merge.cuh"

namespace pkv {

namespace {

constexpr int kMergeWarps = 4;

template <int D>
__global__ void __launch_bounds__(kMergeWarps * 32)
    merge_kernel(pkv_workspace ws, int batch, int S, int flags) {
  __shared__ int s_max_len;
  // Splits past a request's end were never written: merge only the first
  // ceil(L_b / chunk), with chunk derived exactly as the attention kernel did.
  const int chunk = split_chunk(batch_max_len(ws, batch, &s_max_len), S, ws.page_size);
  const int lane = threadIdx.x & 31;
  const long long wg = (long long)blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
  if (wg >= (long long)batch * ws.n_q_heads) return;
  const int n = min(S, split_count(ws, (int)(wg / ws.n_q_heads), chunk));
  float M, den;
  float4 acc;
  merge_row<D>(ws.ml_part + wg * S * 2, ws.o_part + wg * S * D, n, lane, M, den, acc);
  merge_store<D>(ws, wg, flags, lane, M, den, acc);
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
