// Work decomposition shared by the decode kernels.
//
// Unit u in [0, S * B * Hkv) is (split c, request b, KV head g) with
// c = u / (B*Hkv): all first splits come first, so a persistent grid striding
// over u spreads every request's splits across CTAs.  Split c of request b
// covers tokens [c*chunk, min((c+1)*chunk, L_b)); chunk comes from the live
// maximum length (split_chunk), so no request needs more than S splits.
#pragma once

#include "common.cuh"

namespace pkv {

struct Plan {
  int batch, hkv, S, chunk, n_units;
};

struct Unit {
  int u, b, g, c, t0, t1;
};

__device__ __forceinline__ Unit unit_at(const pkv_workspace &ws, const Plan &pl, int u) {
  Unit x;
  x.u = u;
  const int hb = pl.batch * pl.hkv;
  x.c = u / hb;
  const int r = u - x.c * hb;
  x.b = r / pl.hkv;
  x.g = r - x.b * pl.hkv;
  int L = ws.seq_lens[x.b];
  const long long cap = (long long)ws.max_pages_per_req * ws.page_size;
  if (L < 0 || (long long)L > cap) L = 0;  // flagged by the prologue of CTA 0
  if (ws.index_mode == PKV_IDX_FLAT && L > 0) {
    const int base = ws.kv_indptr[x.b];
    if (base < 0 || (long long)base + L > ws.max_total_tokens) L = 0;
  }
  x.t0 = x.c * pl.chunk;
  x.t1 = min(x.t0 + pl.chunk, L);
  return x;
}

// Cursor over a CTA's stream of tiles of TILE tokens (uniform in a warp).
template <int TILE>
struct Cursor {
  Unit un;
  int i;       // next tile of un
  int ntiles;  // tiles of un
  bool done;

  __device__ __forceinline__ void seek(const pkv_workspace &ws, const Plan &pl, int u) {
    for (; u < pl.n_units; u += gridDim.x) {
      un = unit_at(ws, pl, u);
      if (un.t0 < un.t1) {
        i = 0;
        ntiles = (un.t1 - un.t0 + TILE - 1) / TILE;
        done = false;
        return;
      }
    }
    done = true;
  }
  __device__ __forceinline__ void advance(const pkv_workspace &ws, const Plan &pl) {
    if (++i == ntiles) seek(ws, pl, un.u + gridDim.x);
  }
};

// Block prologue: the longest valid length of the batch (CTA 0 also raises
// the length error bits).  Every thread of the block must call it.
__device__ __forceinline__ int batch_max_len(const pkv_workspace &ws, int batch, int *s_max) {
  if (threadIdx.x == 0) *s_max = 0;
  __syncthreads();
  int mx = 0;
  const long long cap = (long long)ws.max_pages_per_req * ws.page_size;
  for (int b = threadIdx.x; b < batch; b += blockDim.x) {
    const int L = ws.seq_lens[b];
    if (L >= 0 && (long long)L <= cap) mx = max(mx, L);
    else if (blockIdx.x == 0) atomicOr(ws.err, PKV_DEVERR_LEN);
    if (blockIdx.x == 0 && ws.index_mode == PKV_IDX_FLAT && L > 0) {
      const int base = ws.kv_indptr[b];
      if (base < 0 || (long long)base + L > ws.max_total_tokens) atomicOr(ws.err, PKV_DEVERR_TOTAL);
    }
  }
  mx = __reduce_max_sync(0xffffffffu, mx);
  if ((threadIdx.x & 31) == 0) atomicMax(s_max, mx);
  __syncthreads();
  return *s_max;
}

// Slot of token `tok` of request b, or -1 with *kind set to the error bit.
__device__ __forceinline__ long long token_slot(const pkv_workspace &ws, int b, int tok,
                                                int &kind) {
  if (ws.index_mode == PKV_IDX_FLAT) {
    const int s = ws.kv_indices[ws.kv_indptr[b] + tok];
    if (s >= 0 && s < ws.pool_slots) return s;
    kind = PKV_DEVERR_SLOT;
    return -1;
  }
  const int row = ws.req_pool_indices[b];
  if (row < 0 || row >= ws.max_reqs) {
    kind = PKV_DEVERR_PAGE;
    return -1;
  }
  const int P = ws.page_size;
  const int page = ws.page_table[(long long)row * ws.max_pages_per_req + tok / P];
  if (page >= 0 && page < ws.pool_slots / P) return (long long)page * P + tok % P;
  kind = PKV_DEVERR_PAGE;
  return -1;
}

}  // namespace pkv
