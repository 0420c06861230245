// Work decomposition of the tensor-core decode kernel.
//
// Fixed chunks: unit u in [0, S * B * Hkv) is (split c, request b, KV head g)
// with c = u / (B*Hkv): all first splits come first, so a persistent grid
// striding over u spreads every request's splits across CTAs.  Split c of
// request b covers tokens [c*chunk, min((c+1)*chunk, L_b)); chunk comes from
// the live maximum length (split_chunk), so no request needs more than S
// splits.  Compact enumeration skips the splits past each request's end.
//
// Apportioned splits (fused merge only): the resident blocks are shared out
// among the requests in proportion to their lengths, request b getting n_b
// splits of one per-request chunk (a multiple of kChunkAlign tokens) for each
// of its KV heads, with Hkv * sum n_b never above the blocks: every block
// then has at most one unit, and the units are as even as whole tiles allow
// whatever the length mix.
#pragma once

#include "common.cuh"

namespace pkv {

struct Plan {
  int batch, hkv, S, chunk, n_units;
  // Compact enumeration: exclusive prefix over requests of their split counts
  // and their usable lengths (shared memory, batch + 1 / batch entries);
  // NULL = dense enumeration.
  // Apportioned splits: chunks[b] is request b's chunk (else NULL: the one
  // chunk above).
  const int *pref = nullptr;
  const int *lens = nullptr;
  const int *chunks = nullptr;
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

// Layout of ws.work_plan (int32 offsets), written by the step's plan kernel
// and read by the decode kernel: a header, the compact plan's arrays, and the
// TMA page ids of the first kPlanTiles tiles of every block.
constexpr int kPlanMagic = 0x706b7631;
constexpr int kPlanTiles = 8;
constexpr int kPlanMaxGrid = 1024;
enum PlanHdr { kHMagic, kHBatch, kHSplits, kHGrid, kHUnits, kHChunk, kHMaxLen, kHApportion,
               kHTma, kHHkv, kPlanHdr = 16 };
constexpr int kPlanPref = kPlanHdr;                          // batch + 1 entries
constexpr int kPlanLen = kPlanPref + kMaxCompactBatch + 4;
constexpr int kPlanBase = kPlanLen + kMaxCompactBatch;
constexpr int kPlanChunk = kPlanBase + kMaxCompactBatch;
constexpr int kPlanFirst = kPlanChunk + kMaxCompactBatch;    // [block][tile][4]
constexpr int kPlanInts = kPlanFirst + kPlanMaxGrid * kPlanTiles * 4;
constexpr int kChunkAlign = 64;  // apportioned chunks: multiples of this many tokens
constexpr int kMinChunk = 128;   // no apportioned split shorter (more merging than streaming)

struct Unit {
  int u, b, g, c, t0, t1;
  int L;  // the request's (checked) length
  int n;  // splits (pieces) of this (request, KV head) that produce a partial
};

// Length of request b as the kernels use it (0 if out of range).
__device__ __forceinline__ int usable_len(const pkv_workspace &ws, int b) {
  int L = ws.seq_lens[b];
  const long long cap = len_cap(ws);
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
    x.n = pl.pref[lo + 1] - pl.pref[lo];
  } else {
    const int hb = pl.batch * pl.hkv;
    x.c = u / hb;
    const int r = u - x.c * hb;
    x.b = r / pl.hkv;
    x.g = r - x.b * pl.hkv;
  }
  x.L = pl.lens ? pl.lens[x.b] : usable_len(ws, x.b);  // bad lengths flagged by CTA 0
  const int chunk = pl.chunks ? pl.chunks[x.b] : pl.chunk;
  x.t0 = x.c * chunk;
  x.t1 = min(x.t0 + chunk, x.L);
  if (!pl.pref) x.n = x.L > 0 ? (x.L + chunk - 1) / chunk : 0;
  return x;
}

// The units block blk of nblk processes, in order (uniform in the block):
// every nblk-th unit from blk, empty ones included.
struct UnitIter {
  Unit un;
  bool done;
  int nblk;

  __device__ __forceinline__ void at(const pkv_workspace &ws, const Plan &pl, int u) {
    done = u >= pl.n_units;
    if (!done) un = unit_at(ws, pl, u);
  }
  __device__ __forceinline__ void first(const pkv_workspace &ws, const Plan &pl, int blk,
                                        int n) {
    nblk = n;
    at(ws, pl, blk);
  }
  __device__ __forceinline__ void first(const pkv_workspace &ws, const Plan &pl) {
    first(ws, pl, blockIdx.x, gridDim.x);
  }
  __device__ __forceinline__ void next(const pkv_workspace &ws, const Plan &pl) {
    at(ws, pl, un.u + nblk);
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
  // as block blk of a grid of n
  __device__ __forceinline__ void start(const pkv_workspace &ws, const Plan &pl, int blk, int n) {
    it.first(ws, pl, blk, n);
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
  const long long cap = len_cap(ws);
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

// Apportioned splits: the search for the common split length X (a multiple
// of kChunkAlign, at least kMinChunk and maxL / S) starts from the even share
// Hkv * sum L / budget and grows by about 1/16 per step until
// Hkv * sum ceil(L_b / X) fits the budget (bounded: after kSearchSteps steps,
// or past the longest request, X is one split per request).  Request b's own chunk then evens its
// ceil(L_b / X) splits out: ceil(L_b / n_b) rounded up to kChunkAlign.
constexpr int kSearchSteps = 48;

__device__ __forceinline__ int align_chunk(long long c) {
  return (int)((c + kChunkAlign - 1) / kChunkAlign * kChunkAlign);
}

__device__ __forceinline__ int apportion_start(long long sum_len, int max_len, int hkv,
                                               int budget, int S) {
  // the even share (a float estimate is enough: the search only grows it)
  long long x = (long long)__fdividef((float)hkv * (float)sum_len, (float)budget);
  x = max(x, (long long)(max_len + S - 1) / S);
  return max(align_chunk(x), kMinChunk);
}

__device__ __forceinline__ int apportion_step(int x) {
  return x + max(kChunkAlign, align_chunk(x / 16));
}

__device__ __forceinline__ int apportioned_chunk(int L, int x) {
  const int n = (L + x - 1) / x;
  return align_chunk((L + n - 1) / n);
}

// Block prologue for compact enumeration (batch <= kMaxCompactBatch): one
// pass reads every request's usable length into s_len (CTA 0 raises the
// length error bits) and its index base into s_base (the table row in page
// mode, the kv_indptr offset in flat mode); the split counts then follow from
// shared memory and their exclusive prefix goes to s_pref.  budget == 0:
// fixed chunks (one chunk from the longest length and S); budget > 0:
// apportioned splits over `budget` blocks, each request's chunk in s_chunk.
// Every thread of the block must call it; returns the number of non-empty
// (request, split) pairs and sets *chunk_out (the longest usable length stays
// in *s_max).
__device__ __forceinline__ int batch_plan_compact(const pkv_workspace &ws, int batch, int S,
                                                  int budget, int *s_len, int *s_base,
                                                  int *s_pref, int *s_chunk, int *s_tmp,
                                                  int *s_max, int *chunk_out) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int hkv = ws.n_kv_heads;
  const long long cap = len_cap(ws);
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
  // splits of request b (length L): fixed chunks, or apportioned with split
  // length x (recording its chunk)
  auto splits = [&](int b, int L, int chunk, int x) {
    if (L <= 0) return 0;
    if (budget == 0) return (L + chunk - 1) / chunk;
    const int c = apportioned_chunk(L, x);
    s_chunk[b] = c;
    return (L + c - 1) / c;
  };
  if (batch <= 32) {
    // one warp: sums, maximum and prefix by shuffles, one block barrier
    if (warp == 0) {
      const int L = lane < batch ? read_req(lane) : 0;
      const int mx = __reduce_max_sync(0xffffffffu, L);
      const int chunk = split_chunk(mx, S, ws.page_size);
      int x = 0;
      if (budget > 0 && mx > 0) {
        const long long sum_len = __reduce_add_sync(0xffffffffu, (unsigned)L);
        x = apportion_start(sum_len, mx, hkv, budget, S);
        for (int step = 0; x < mx; ++step, x = apportion_step(x)) {
          const int n = L > 0 ? (L + x - 1) / x : 0;
          if ((long long)hkv * __reduce_add_sync(0xffffffffu, (unsigned)n) <= budget) break;
          if (step == kSearchSteps) {
            x = align_chunk(mx);
            break;
          }
        }
      }
      const int cnt = splits(lane, L, chunk, x);
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
  if (tid == 0) {
    *s_max = 0;
    s_tmp[0] = 0;  // sum of the lengths
  }
  __syncthreads();
  int mx = 0, sum = 0;
  for (int b = tid; b < batch; b += blockDim.x) {
    const int L = read_req(b);
    mx = max(mx, L);
    sum += L;
  }
  mx = __reduce_max_sync(0xffffffffu, mx);
  sum = (int)__reduce_add_sync(0xffffffffu, (unsigned)sum);
  if (lane == 0) {
    atomicMax(s_max, mx);
    atomicAdd(&s_tmp[0], sum);
  }
  __syncthreads();
  const int chunk = split_chunk(*s_max, S, ws.page_size);
  *chunk_out = chunk;
  int x = 0;
  const int mxl = *s_max;
  if (budget > 0 && mxl > 0) {
    x = apportion_start(s_tmp[0], mxl, hkv, budget, S);
    __syncthreads();  // everyone has read s_tmp[0]
    for (int step = 0; x < mxl; ++step, x = apportion_step(x)) {
      int n = 0;
      for (int b = tid; b < batch; b += blockDim.x) n += (s_len[b] + x - 1) / x;
      n = (int)__reduce_add_sync(0xffffffffu, (unsigned)n);
      if (tid == 0) s_tmp[2 + (step & 1)] = 0;  // this step's counter (the other one was last read a barrier ago)
      __syncthreads();
      if (lane == 0) atomicAdd(&s_tmp[2 + (step & 1)], n);
      __syncthreads();
      const bool fits = (long long)hkv * s_tmp[2 + (step & 1)] <= budget;
      if (fits) break;
      if (step == kSearchSteps) {
        x = align_chunk(mxl);
        break;
      }
    }
    __syncthreads();  // s_tmp is reused by the scan below
  }
  const int nt = blockDim.x;
  const int per = (batch + nt - 1) / nt;
  const int lo = min(batch, tid * per), hi = min(batch, lo + per);
  int local = 0;
  for (int b = lo; b < hi; ++b) local += splits(b, s_len[b], chunk, x);
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
    run += (s_len[b] <= 0) ? 0
           : (budget == 0 ? (s_len[b] + chunk - 1) / chunk
                          : (s_len[b] + s_chunk[b] - 1) / s_chunk[b]);
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
