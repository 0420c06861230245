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
  // Compact enumeration: exclusive prefix over requests of their split counts
  // and their usable lengths (shared memory, batch + 1 / batch entries);
  // NULL = dense enumeration.
  const int *pref = nullptr;
  const int *lens = nullptr;
};

constexpr int kMaxCompactBatch = 512;

struct Unit {
  int u, b, g, c, t0, t1;
  int L;  // the request's (checked) length
};

// Length of request b as the kernels use it (0 if out of range).
__device__ __forceinline__ int usable_len(const pkv_workspace &ws, int b) {
  int L = ws.seq_lens[b];
  const long long cap = (long long)ws.max_pages_per_req * ws.page_size;
  if (L < 0 || (long long)L > cap) return 0;
  if (ws.index_mode == PKV_IDX_FLAT && L > 0) {
    const int base = ws.kv_indptr[b];
    if (base < 0 || (long long)base + L > ws.max_total_tokens) return 0;
  }
  return L;
}

__device__ __forceinline__ int split_count(const pkv_workspace &ws, int b, int chunk) {
  const int L = usable_len(ws, b);
  return L > 0 ? (L + chunk - 1) / chunk : 0;
}

__device__ __forceinline__ Unit unit_at(const pkv_workspace &ws, const Plan &pl, int u) {
  Unit x;
  x.u = u;
  if (pl.pref) {
    // u = (pair, g) over the non-empty (request, split) pairs in request order.
    const int w = u / pl.hkv;
    x.g = u - w * pl.hkv;
    int lo = 0, hi = pl.batch - 1;  // last b with pref[b] <= w
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pl.pref[mid] <= w) lo = mid;
      else hi = mid - 1;
    }
    x.b = lo;
    x.c = w - pl.pref[lo];
  } else {
    const int hb = pl.batch * pl.hkv;
    x.c = u / hb;
    const int r = u - x.c * hb;
    x.b = r / pl.hkv;
    x.g = r - x.b * pl.hkv;
  }
  x.L = pl.lens ? pl.lens[x.b] : usable_len(ws, x.b);  // bad lengths flagged by CTA 0
  x.t0 = x.c * pl.chunk;
  x.t1 = min(x.t0 + pl.chunk, x.L);
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

// Block-wide exclusive prefix of the requests' split counts into
// s_pref[0..batch] (batch <= kMaxCompactBatch); s_tmp holds 32 ints.  Every
// thread of the block must call it; returns the number of non-empty
// (request, split) pairs.
__device__ __forceinline__ int batch_split_prefix(const pkv_workspace &ws, int batch, int chunk,
                                                  int *s_pref, int *s_tmp) {
  const int nt = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (batch + nt - 1) / nt;
  const int lo = min(batch, tid * per), hi = min(batch, lo + per);
  int local = 0;
  for (int b = lo; b < hi; ++b) local += split_count(ws, b, chunk);
  int incl = local;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31) s_tmp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < (nt + 31) / 32 ? s_tmp[lane] : 0;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, w, d);
      if (lane >= d) w += v;
    }
    s_tmp[lane] = w;
  }
  __syncthreads();
  int run = (warp > 0 ? s_tmp[warp - 1] : 0) + incl - local;
  for (int b = lo; b < hi; ++b) {
    s_pref[b] = run;
    run += split_count(ws, b, chunk);
  }
  if (tid == nt - 1) s_pref[batch] = run;
  __syncthreads();
  return s_pref[batch];
}

// Block prologue for compact enumeration (batch <= kMaxCompactBatch): one
// pass reads every request's usable length into s_len (CTA 0 raises the
// length error bits) and its index base into s_base (the table row in page
// mode, the kv_indptr offset in flat mode), then the split length and the
// exclusive prefix of the split counts follow from shared memory.  Every thread of the block must
// call it; returns the number of non-empty (request, split) pairs and sets
// *chunk_out.
__device__ __forceinline__ int batch_plan_compact(const pkv_workspace &ws, int batch, int S,
                                                  int *s_len, int *s_base, int *s_pref,
                                                  int *s_tmp, int *s_max, int *chunk_out) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) *s_max = 0;
  __syncthreads();
  int mx = 0;
  const long long cap = (long long)ws.max_pages_per_req * ws.page_size;
  for (int b = tid; b < batch; b += blockDim.x) {
    const int raw = ws.seq_lens[b];
    s_base[b] = ws.index_mode == PKV_IDX_FLAT ? ws.kv_indptr[b] : ws.req_pool_indices[b];
    int L = raw;
    if (L < 0 || (long long)L > cap) {
      if (blockIdx.x == 0) atomicOr(ws.err, PKV_DEVERR_LEN);
      L = 0;
    } else if (ws.index_mode == PKV_IDX_FLAT && L > 0) {
      const int base = ws.kv_indptr[b];
      if (base < 0 || (long long)base + L > ws.max_total_tokens) {
        if (blockIdx.x == 0) atomicOr(ws.err, PKV_DEVERR_TOTAL);
        L = 0;
      }
    }
    s_len[b] = L;
    mx = max(mx, L);
  }
  mx = __reduce_max_sync(0xffffffffu, mx);
  if (lane == 0) atomicMax(s_max, mx);
  __syncthreads();
  const int chunk = split_chunk(*s_max, S, ws.page_size);
  *chunk_out = chunk;
  const int nt = blockDim.x;
  const int per = (batch + nt - 1) / nt;
  const int lo = min(batch, tid * per), hi = min(batch, lo + per);
  int local = 0;
  for (int b = lo; b < hi; ++b) local += (s_len[b] + chunk - 1) / chunk;
  int incl = local;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31) s_tmp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < (nt + 31) / 32 ? s_tmp[lane] : 0;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, w, d);
      if (lane >= d) w += v;
    }
    s_tmp[lane] = w;
  }
  __syncthreads();
  int run = (warp > 0 ? s_tmp[warp - 1] : 0) + incl - local;
  for (int b = lo; b < hi; ++b) {
    s_pref[b] = run;
    run += (s_len[b] + chunk - 1) / chunk;
  }
  if (tid == nt - 1) s_pref[batch] = run;
  __syncthreads();
  return s_pref[batch];
}

// Where a request's index entries start: the table row (page mode) or the
// kv_indptr offset (flat mode).  ok = false for a table row out of range.
struct ReqIndex {
  long long base;
  bool ok;
};

// As req_index, from the bases cached by batch_plan_compact.
__device__ __forceinline__ ReqIndex req_index_cached(const pkv_workspace &ws, const int *s_base,
                                                     int b) {
  ReqIndex r;
  if (ws.index_mode == PKV_IDX_FLAT) {
    r.base = s_base[b];
    r.ok = true;
  } else {
    const int row = s_base[b];
    r.ok = row >= 0 && row < ws.max_reqs;
    r.base = r.ok ? (long long)row * ws.max_pages_per_req : 0;
  }
  return r;
}

__device__ __forceinline__ ReqIndex req_index(const pkv_workspace &ws, int b) {
  ReqIndex r;
  if (ws.index_mode == PKV_IDX_FLAT) {
    r.base = ws.kv_indptr[b];
    r.ok = true;  // usable_len already checked the range against max_total_tokens
  } else {
    const int row = ws.req_pool_indices[b];
    r.ok = row >= 0 && row < ws.max_reqs;
    r.base = r.ok ? (long long)row * ws.max_pages_per_req : 0;
  }
  return r;
}

// Raw index entry of token tok (flat: its slot; page mode: its page id).
__device__ __forceinline__ int raw_index(const pkv_workspace &ws, const ReqIndex &ri, int tok) {
  if (!ri.ok) return -1;
  return ws.index_mode == PKV_IDX_FLAT ? ws.kv_indices[ri.base + tok]
                                       : ws.page_table[ri.base + tok / ws.page_size];
}

// Slot from a raw entry, or -1 with *kind set to the error bit.
__device__ __forceinline__ long long slot_from_raw(const pkv_workspace &ws, int raw, int tok,
                                                   int &kind) {
  if (ws.index_mode == PKV_IDX_FLAT) {
    if (raw >= 0 && raw < ws.pool_slots) return raw;
    kind = PKV_DEVERR_SLOT;
    return -1;
  }
  const int P = ws.page_size;
  if (raw >= 0 && raw < ws.pool_slots / P) return (long long)raw * P + tok % P;
  kind = PKV_DEVERR_PAGE;
  return -1;
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
