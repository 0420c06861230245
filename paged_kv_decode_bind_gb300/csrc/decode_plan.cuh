// Work decomposition of the tensor-core decode kernel.
//
// Fixed chunks: unit u in [0, S * B * Hkv) is (split c, request b, KV head g)
// with c = u / (B*Hkv): all first splits come first, so a persistent grid
// striding over u spreads every request's splits across CTAs.  Split c of
// request b covers tokens [c*chunk, min((c+1)*chunk, L_b)); chunk comes from
// the live maximum length (split_chunk), so no request needs more than S
// splits.  Compact enumeration skips the splits past each request's end.
//
// Balanced pieces (fused merge only): the (request, KV head) segments of the
// batch are laid end to end, b-major, and block i takes the positions
// [i*W, (i+1)*W) of that line, W = ceil(T / blocks) for T positions in all;
// inside a segment the cut points are rounded up to a multiple of
// kPieceAlign tokens.  Every block then streams the same number of tokens
// (to within a tile per segment it touches) whatever the length mix, and a
// segment's pieces are its splits, numbered from 0 in token order.
#pragma once

#include "common.cuh"

namespace pkv {

struct Plan {
  int batch, hkv, S, chunk, n_units;
  // Compact enumeration: exclusive prefix over requests of their split counts
  // and their usable lengths (shared memory, batch + 1 / batch entries);
  // NULL = dense enumeration.
  // Balanced pieces: pref is the exclusive prefix of the usable lengths,
  // W the positions per block, T = hkv * pref[batch].
  // Both fit in 31 bits (the launcher checks Hkv * batch * capacity).
  const int *pref = nullptr;
  const int *lens = nullptr;
  bool balanced = false;
  int W = 0, T = 0;
  // Page geometry, so that the per-tile index arithmetic needs no division
  // when the page size is a power of two.
  int P = 1, pshift = 0, n_pages = 0;

  __device__ __forceinline__ void set_pages(const pkv_workspace &ws) {
    P = ws.page_size;
    pshift = (P & (P - 1)) == 0 ? __ffs(P) - 1 : -1;
    n_pages = ws.pool_slots / P;
  }
  __device__ __forceinline__ int page_of(int tok) const {
    return pshift >= 0 ? tok >> pshift : tok / P;
  }
  __device__ __forceinline__ int in_page(int tok) const {
    return pshift >= 0 ? tok & (P - 1) : tok - (tok / P) * P;
  }
};

constexpr int kMaxCompactBatch = 256;
constexpr int kPieceAlign = 64;  // balanced cut points: multiples of this many tokens
constexpr int kMinPiece = 128;   // balanced share floor: shorter pieces cost more to merge

struct Unit {
  int u, b, g, c, t0, t1;
  int L;  // the request's (checked) length
  int n;  // splits (pieces) of this (request, KV head) that produce a partial
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
  x.n = x.L > 0 ? (x.L + pl.chunk - 1) / pl.chunk : 0;
  return x;
}

// Balanced pieces: cut point at line position x inside a segment of L tokens.
__device__ __forceinline__ int piece_edge(long long x, int L) {
  if (x <= 0) return 0;
  const long long r = (x + kPieceAlign - 1) / kPieceAlign * kPieceAlign;
  return r < L ? (int)r : L;
}

// This block's piece of segment (b, g) (empty if the rounded cut points meet).
// The segment starts at line position o inside block o / W's range, which
// owns its piece 0; the piece count follows from the last cut point below L.
__device__ __forceinline__ Unit piece_at(const Plan &pl, int b, int g) {
  Unit x;
  x.b = b;
  x.g = g;
  x.u = b * pl.hkv + g;
  x.L = pl.lens[b];
  const int o = pl.hkv * pl.pref[b] + g * x.L;  // < T
  const long long lo = (long long)blockIdx.x * pl.W;
  x.t0 = piece_edge(lo - o, x.L);
  x.t1 = piece_edge(lo + pl.W - o, x.L);
  const int first = o / pl.W;
  x.c = (int)blockIdx.x - first;
  const int last_cut = (x.L - 1) / kPieceAlign * kPieceAlign;
  x.n = (o + last_cut) / pl.W - first + 1;  // o + last_cut < T
  return x;
}

// The units one block processes, in order (uniform in the block).  Fixed
// chunks: every gridDim.x-th unit, empty ones included; balanced pieces: the
// non-empty pieces of the segments meeting the block's range.
struct UnitIter {
  Unit un;
  bool done;

  __device__ __forceinline__ void strided(const pkv_workspace &ws, const Plan &pl, int u) {
    done = u >= pl.n_units;
    if (!done) un = unit_at(ws, pl, u);
  }
  __device__ __forceinline__ void first(const pkv_workspace &ws, const Plan &pl) {
    if (!pl.balanced) {
      strided(ws, pl, blockIdx.x);
      return;
    }
    const long long lo = (long long)blockIdx.x * pl.W;
    done = lo >= pl.T;
    if (done) return;
    // the request holding position lo: the last b with hkv * pref[b] <= lo
    // (its length is > 0 because lo < T)
    int l = 0, h = pl.batch - 1;
    while (l < h) {
      const int mid = (l + h + 1) >> 1;
      if (pl.hkv * pl.pref[mid] <= lo) l = mid;
      else h = mid - 1;
    }
    const int L = pl.lens[l];
    if (L <= 0) {
      done = true;
      return;
    }
    un = piece_at(pl, l, ((int)lo - pl.hkv * pl.pref[l]) / L);
    // only the first segment's piece can be empty (its cut points rounded
    // past the segment's end: the next block owns that tail)
    if (un.t0 >= un.t1) next(ws, pl);
  }
  __device__ __forceinline__ void next(const pkv_workspace &ws, const Plan &pl) {
    if (!pl.balanced) {
      strided(ws, pl, un.u + gridDim.x);
      return;
    }
    int b = un.b, g = un.g + 1;
    if (g == pl.hkv) {
      g = 0;
      do ++b;
      while (b < pl.batch && pl.lens[b] == 0);
    }
    done = b >= pl.batch ||
           pl.hkv * pl.pref[b] + g * pl.lens[b] >= (long long)(blockIdx.x + 1) * pl.W;
    if (!done) un = piece_at(pl, b, g);
  }
};

// Cursor over a CTA's stream of tiles of TILE tokens (uniform in a warp):
// the tiles of its non-empty units, in order.
template <int TILE>
struct Cursor {
  UnitIter it;
  int i;       // next tile of it.un
  int ntiles;  // tiles of it.un
  bool done;

  __device__ __forceinline__ void skip_empty(const pkv_workspace &ws, const Plan &pl) {
    while (!it.done && it.un.t0 >= it.un.t1) it.next(ws, pl);
    done = it.done;
    if (!done) {
      i = 0;
      ntiles = (it.un.t1 - it.un.t0 + TILE - 1) / TILE;
    }
  }
  __device__ __forceinline__ void start(const pkv_workspace &ws, const Plan &pl) {
    it.first(ws, pl);
    skip_empty(ws, pl);
  }
  __device__ __forceinline__ void advance(const pkv_workspace &ws, const Plan &pl) {
    if (++i == ntiles) {
      it.next(ws, pl);
      skip_empty(ws, pl);
    }
  }
  // n >= 0 tiles further (past the end: done)
  __device__ __forceinline__ void advance_by(const pkv_workspace &ws, const Plan &pl, int n) {
    while (n > 0 && !done) {
      const int take = min(n, ntiles - i);
      i += take;
      n -= take;
      if (i == ntiles) {
        it.next(ws, pl);
        skip_empty(ws, pl);
      }
    }
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

// Block prologue for compact enumeration (batch <= kMaxCompactBatch): one
// pass reads every request's usable length into s_len (CTA 0 raises the
// length error bits) and its index base into s_base (the table row in page
// mode, the kv_indptr offset in flat mode), then the split length and an
// exclusive prefix into s_pref follow from shared memory: of the split counts
// (fixed chunks), or of the lengths themselves (by_len, balanced pieces).
// Every thread of the block must call it; returns s_pref[batch] and sets
// *chunk_out (the longest usable length stays in *s_max).
__device__ __forceinline__ int batch_plan_compact(const pkv_workspace &ws, int batch, int S,
                                                  bool by_len, int *s_len, int *s_base,
                                                  int *s_pref, int *s_tmp, int *s_max,
                                                  int *chunk_out) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long cap = (long long)ws.max_pages_per_req * ws.page_size;
  // request b's usable length (and its index base into s_base[b])
  auto read_req = [&](int b) {
    const int raw = ws.seq_lens[b];
    const int base = ws.index_mode == PKV_IDX_FLAT ? ws.kv_indptr[b] : ws.req_pool_indices[b];
    s_base[b] = base;
    int L = raw;
    if (L < 0 || (long long)L > cap) {
      if (blockIdx.x == 0) atomicOr(ws.err, PKV_DEVERR_LEN);
      L = 0;
    } else if (ws.index_mode == PKV_IDX_FLAT && L > 0 &&
               (base < 0 || (long long)base + L > ws.max_total_tokens)) {
      if (blockIdx.x == 0) atomicOr(ws.err, PKV_DEVERR_TOTAL);
      L = 0;
    }
    s_len[b] = L;
    return L;
  };
  if (batch <= 32) {
    // one warp: maximum and prefix by shuffles, one block barrier
    if (warp == 0) {
      const int L = lane < batch ? read_req(lane) : 0;
      const int mx = __reduce_max_sync(0xffffffffu, L);
      const int chunk = split_chunk(mx, S, ws.page_size);
      const int cnt = by_len ? L : (L + chunk - 1) / chunk;
      int incl = cnt;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += v;
      }
      if (lane < batch) s_pref[lane] = incl - cnt;
      if (lane == 31) {
        s_pref[batch] = incl;  // lanes past the batch add nothing
        *s_max = mx;
        s_tmp[0] = chunk;
      }
    }
    __syncthreads();
    *chunk_out = s_tmp[0];
    return s_pref[batch];
  }
  if (tid == 0) *s_max = 0;
  __syncthreads();
  int mx = 0;
  for (int b = tid; b < batch; b += blockDim.x) mx = max(mx, read_req(b));
  mx = __reduce_max_sync(0xffffffffu, mx);
  if (lane == 0) atomicMax(s_max, mx);
  __syncthreads();
  const int chunk = split_chunk(*s_max, S, ws.page_size);
  *chunk_out = chunk;
  const int nt = blockDim.x;
  const int per = (batch + nt - 1) / nt;
  const int lo = min(batch, tid * per), hi = min(batch, lo + per);
  auto count = [&](int b) { return by_len ? s_len[b] : (s_len[b] + chunk - 1) / chunk; };
  int local = 0;
  for (int b = lo; b < hi; ++b) local += count(b);
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
    run += count(b);
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

// Where the raw index entry of token tok of a request lives (its request's
// entries start at ri.base; ri.ok).
__device__ __forceinline__ const int *index_src(const pkv_workspace &ws, const Plan &pl,
                                                const ReqIndex &ri, int tok) {
  return ws.index_mode == PKV_IDX_FLAT ? ws.kv_indices + ri.base + tok
                                       : ws.page_table + ri.base + pl.page_of(tok);
}

// Slot from a raw entry, or -1 with *kind set to the error bit.
__device__ __forceinline__ long long slot_from_raw(const pkv_workspace &ws, const Plan &pl,
                                                   int raw, int tok, int &kind) {
  if (ws.index_mode == PKV_IDX_FLAT) {
    if (raw >= 0 && raw < ws.pool_slots) return raw;
    kind = PKV_DEVERR_SLOT;
    return -1;
  }
  if (raw >= 0 && raw < pl.n_pages) return (long long)raw * pl.P + pl.in_page(tok);
  kind = PKV_DEVERR_PAGE;
  return -1;
}

}  // namespace pkv
