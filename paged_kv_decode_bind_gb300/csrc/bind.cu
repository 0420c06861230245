// Per-step decode metadata and KV append (cache.py page, bullets 25, 26, 28
// and 40; workspace.py page, bullet 24).
//
//   bind_meta_kernel    one CTA: new seq_lens, position_ids, the exclusive
//                       prefix sum kv_indptr and out_loc, in place.
//   flat_index_kernel   flat mode: kv_indices[kv_indptr[b] + t] =
//                       request-to-token table row of b, for t < seq_lens[b].
//   append_kernel       pool[layer, out_loc[b]] = new row, for K and V.
#include "kernels.cuh"

namespace pkv {

namespace {

constexpr int kMetaThreads = 1024;
constexpr int kMetaPer = 8;  // batch entries per thread -> max_batch <= 8192

__global__ void __launch_bounds__(kMetaThreads) bind_meta_kernel(pkv_workspace ws, int batch,
                                                                 int mode) {
  __shared__ long long s_warp[kMetaThreads / 32];
  const int tid = threadIdx.x;
  const int per = (batch + kMetaThreads - 1) / kMetaThreads;
  const int lo = tid * per;
  const long long cap = len_cap(ws);

  int old_len[kMetaPer];
  int new_len[kMetaPer];
  long long local = 0;
#pragma unroll
  for (int i = 0; i < kMetaPer; ++i) {
    const int b = lo + i;
    old_len[i] = 0;
    new_len[i] = 0;
    if (i < per && b < batch) {
      old_len[i] = ws.seq_lens[b];
      new_len[i] = mode == PKV_BIND_STEADY ? old_len[i] + 1 : old_len[i];
      local += new_len[i] > 0 ? new_len[i] : 0;
    }
  }

  // Block-wide exclusive scan of the per-thread sums.
  const int lane = tid & 31, warp = tid >> 5;
  long long incl = local;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const long long v = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();  // every read of seq_lens above happens before any write below
  if (warp == 0) {
    long long w = s_warp[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const long long v = __shfl_up_sync(0xffffffffu, w, d);
      if (lane >= d) w += v;
    }
    s_warp[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  long long run = (warp > 0 ? s_warp[warp - 1] : 0) + incl - local;

  int err = 0;
#pragma unroll
  for (int i = 0; i < kMetaPer; ++i) {
    const int b = lo + i;
    if (!(i < per && b < batch)) continue;
    const int L = new_len[i];
    ws.seq_lens[b] = L;
    ws.position_ids[b] = mode == PKV_BIND_STEADY ? old_len[i] : L - 1;
    if (run > 0x7fffffffll) err |= PKV_DEVERR_TOTAL;
    ws.kv_indptr[b] = (int)run;
    int loc = -1;
    if (L < 0 || (long long)L > cap) {
      err |= PKV_DEVERR_LEN;
    } else if (L > 0) {
      const int row = ws.req_pool_indices[b];
      const int t = L - 1;
      if (row < 0 || row >= ws.max_reqs) {
        err |= PKV_DEVERR_PAGE;
      } else if (ws.index_mode == PKV_IDX_FLAT) {
        const int s = ws.page_table[(long long)row * ws.max_pages_per_req + t];
        if (s < 0 || s >= ws.pool_slots) err |= PKV_DEVERR_SLOT;
        else loc = s;
      } else {
        const int P = ws.page_size;
        const int page = ws.page_table[(long long)row * ws.max_pages_per_req + t / P];
        if (page < 0 || page >= ws.pool_slots / P) err |= PKV_DEVERR_PAGE;
        else loc = page * P + t % P;
      }
    }
    ws.out_loc[b] = loc;
    run += L > 0 ? L : 0;
  }
  if (tid == kMetaThreads - 1) {
    if (run > 0x7fffffffll) err |= PKV_DEVERR_TOTAL;
    ws.kv_indptr[batch] = (int)run;
  }
  if (err) atomicOr(ws.err, err);
}

constexpr int kFlatThreads = 256;

__global__ void __launch_bounds__(kFlatThreads) flat_index_kernel(pkv_workspace ws) {
  const int b = blockIdx.y;
  const int L = ws.seq_lens[b];
  const int base = ws.kv_indptr[b];
  const bool lead = blockIdx.x == 0 && threadIdx.x == 0;
  if (L <= 0) return;
  if ((long long)L > len_cap(ws)) {
    if (lead) atomicOr(ws.err, PKV_DEVERR_LEN);
    return;
  }
  if (base < 0 || (long long)base + L > ws.max_total_tokens) {
    if (lead) atomicOr(ws.err, PKV_DEVERR_TOTAL);
    return;
  }
  const int row = ws.req_pool_indices[b];
  if (row < 0 || row >= ws.max_reqs) {
    if (lead) atomicOr(ws.err, PKV_DEVERR_PAGE);
    return;
  }
  const int *src = ws.page_table + (long long)row * ws.max_pages_per_req;
  int *dst = ws.kv_indices + base;
  int bad = 0;
  for (int t = blockIdx.x * kFlatThreads + threadIdx.x; t < L; t += gridDim.x * kFlatThreads) {
    const int s = src[t];
    bad |= (s < 0 || s >= ws.pool_slots);
    dst[t] = s;
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(ws.err, PKV_DEVERR_SLOT);
}

constexpr int kAppendThreads = 128;

__global__ void __launch_bounds__(kAppendThreads)
    append_kernel(pkv_workspace ws, int batch, int layer_begin, const uint4 *__restrict__ k_new,
                  const uint4 *__restrict__ v_new) {
  const int b = blockIdx.x;
  const int rel = blockIdx.y;
  const int layer = layer_begin + rel;
  const int loc = ws.out_loc[b];
  if (loc < 0 || loc >= ws.pool_slots) {
    if (threadIdx.x == 0) atomicOr(ws.err, PKV_DEVERR_SLOT);
    return;
  }
  const int n16 = ws.n_kv_heads * ws.head_dim / 8;  // 16-byte vectors per row
  const long long dst = ((long long)layer * ws.pool_slots + loc) * n16;
  const long long src = ((long long)rel * batch + b) * n16;
  uint4 *kp = reinterpret_cast<uint4 *>(ws.k_pool);
  uint4 *vp = reinterpret_cast<uint4 *>(ws.v_pool);
  for (int i = threadIdx.x; i < n16; i += kAppendThreads) {
    kp[dst + i] = k_new[src + i];
    vp[dst + i] = v_new[src + i];
  }
}

}  // namespace

cudaError_t launch_bind_meta(const pkv_workspace &ws, int batch, int mode, cudaStream_t st) {
  bind_meta_kernel<<<1, kMetaThreads, 0, st>>>(ws, batch, mode);
  return cudaGetLastError();
}

cudaError_t launch_flat_index(const pkv_workspace &ws, int batch, cudaStream_t st) {
  // Enough blocks per request for ~8k tokens in one pass; longer rows loop.
  const int bx = 32;
  flat_index_kernel<<<dim3(bx, batch), kFlatThreads, 0, st>>>(ws);
  return cudaGetLastError();
}

cudaError_t launch_append(const pkv_workspace &ws, int batch, int layer_begin, int layer_count,
                          const void *k_new, const void *v_new, cudaStream_t st) {
  append_kernel<<<dim3(batch, layer_count), kAppendThreads, 0, st>>>(
      ws, batch, layer_begin, static_cast<const uint4 *>(k_new),
      static_cast<const uint4 *>(v_new));
  return cudaGetLastError();
}

int meta_max_batch() { return kMetaThreads * kMetaPer; }

}  // namespace pkv
