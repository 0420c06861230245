// Tensor-core split-KV GQA decode attention (workspace.py page, bullets 1 and
// 14-16), optionally fused with the KV append (cache.py page, bullet 40) and
// with the split merge.
//
// Math.  Per (request b, KV head g, split c) unit both products keep the
// token axis on the 16-row side of warp-level bf16 mma.m16n8k16 (fp32
// accumulation) and the query group on the 8-wide side, so a group of up to
// 8 heads needs no padding:  S^T = K Q_g^T (16 tokens x 8 heads per k-step of
// 16 dims) and O^T += V^T P^T (16 dims x 8 heads per 16 tokens).  The C
// fragment of S^T becomes the B fragment of P^T with one movmatrix transpose
// per 8x8 block.  P enters as P_hi + P_lo (two bf16 terms) so P V keeps ~16
// mantissa bits.  The K/V rows of a token are read from HBM once for all G
// heads.
//
// Block.  4 consumer warps + 1 producer warp.  A tile is 64 tokens; consumer
// warp w owns tokens [16w, 16w+16) of each tile with its own online-softmax
// state; the four states merge at the end of the unit.  The producer walks
// the block's units ahead of the consumers, across unit boundaries, through a
// 3-stage ring with a `full` and an `empty` mbarrier per stage, fetching
// index entries several tiles ahead (a second cursor, cp.async into a shared
// ring) so their latency overlaps the issue of earlier tiles.
//
// Units.  With batch <= kMaxCompactBatch only the non-empty (request, split)
// pairs are units (a per-block prefix over the requests' split counts), so a
// round-robin over units gives every block the same share.
//
// Shared-memory tile layout: per K (or V) tile, D/64 column halves, each
// [64 rows][128 B] with the 128-byte swizzle (16-byte chunk c of row r sits at
// chunk c ^ (r & 7)), so the 8 row addresses of every ldmatrix hit distinct
// banks.  Two ways fill it:
//   * page mode with P % 16 == 0: the producer issues one tensor-map TMA box
//     per 16-token page piece (both column halves) and pool; `full` completes
//     on the landed bytes, `empty` on the four consumer warps' release;
//   * any other page size and the flat (token-level) mode: the producer
//     validates the tile's index entries into pool slots and publishes them
//     on `full`; each consumer warp then copies its own 16 rows with 16-byte
//     cp.async gathers at the swizzled positions (zero-filled past the end)
//     two tiles ahead of the one it computes, and releases the slots on
//     `empty`.  A single warp issuing all 64 rows' copies was the bottleneck.
//
// Fused append: the unit that holds a request's newest token first writes the
// new K/V row (k_new, v_new) to pool[layer, out_loc[b]], fences the async
// proxy, then loads the tile, so the new token is attended.
// Fused merge: a unit of a request with n > 1 splits writes its partial,
// then takes a ticket on split_counters[b, g]; the unit that draws n - 1
// merges all n partials and resets the counter to 0 (no waiting anywhere).
//
// Every wait is bounded (~1 s); a timeout raises PKV_DEVERR_TIMEOUT, marks the
// unit empty, makes every later wait of the block return at once, and the
// producer drains its copies in flight (again bounded) before exiting.
#include <cuda.h>

#include <cstring>

#include "decode_plan.cuh"
#include "kernels.cuh"
#include "merge.cuh"

namespace pkv {

namespace {

constexpr int kCW = 4;                   // consumer warps
constexpr int kMThreads = (kCW + 1) * 32;
constexpr int kMT = 16 * kCW;            // tokens per tile
constexpr int kMStages = 3;
constexpr int kLA = 8;  // tiles of index lookahead (shared-memory ring of slots)
static_assert(kLA == kPlanTiles, "the step's plan holds the first ring's worth of page ids");

template <int D, int G>
struct MCfg {
  static constexpr int HALVES = D / 64;     // 64-column (128-byte) swizzled halves
  static constexpr int PIECE = 16 * HALVES * 128;  // bytes of a 16-token page piece
  static constexpr int TILE = (kMT / 16) * PIECE;    // bytes of K (or V) of a tile
  static constexpr int KSTEPS = D / 16;
  static constexpr int NH = (G + 7) / 8;    // 8-wide head tiles
  static constexpr int MT = D / 16;         // 16-row output (head_dim) tiles
  static constexpr int RSTRIDE = D + 4;     // combine buffer row stride (floats)
  // dynamic shared memory: the K/V ring (1024-aligned for the swizzle) and
  // the combine buffer; small state lives in static shared memory.
  static constexpr int OFF_KV = 0;
  static constexpr int OFF_RED = OFF_KV + kMStages * 2 * TILE;  // [2][G][RSTRIDE] f32
  static constexpr int SMEM = OFF_RED + 2 * G * RSTRIDE * 4 + 1024;  // + alignment slack
  static_assert(G >= 1 && G <= 16, "one 16-row mma operand per group");
  static_assert(D % 64 == 0, "whole swizzled halves");
};

// Byte offset of 16-byte chunk c (0..7) of 128-byte row r, 128B-swizzled.
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

// A ring stage in shared memory holds, per 16-token page piece, the piece's K
// then its V (the box order of the pool tensor map): each is HALVES x 16 rows
// of 128 bytes, [half][token % 16][64 columns].  Offset of chunk c of token t,
// half h inside the stage's K (or, from the V base, V) data: rows of
// consecutive tokens stay consecutive (conflict-free ldmatrix).
template <int HALVES>
__device__ __forceinline__ uint32_t kv_off(int t, int h, int c) {
  return (uint32_t)((t >> 4) * (2 * 16 * 128 * HALVES)) + swz(h * 16 + (t & 15), c);
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *tm, int c0, int c1,
                                            int c2, int c3, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], "
      "[%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}


// Fused append: write this (request, head)'s new K/V row to the pool when the
// tile [tile0, tile0 + 64) of this unit holds the request's newest token
// (warp-uniform).
template <int D>
__device__ __forceinline__ void append_if_newest(const DecodeArgs &a, const Unit &un, int tile0,
                                                 int lane) {
  if (a.k_new == nullptr || un.L <= 0) return;
  const int t = un.L - 1;
  if (t < tile0 || t >= min(tile0 + kMT, un.t1)) return;
  const pkv_workspace &ws = a.ws;
  const int loc = ws.out_loc[un.b];
  if (loc < 0 || loc >= ws.pool_slots) {
    if (lane == 0) atomicOr(ws.err, PKV_DEVERR_SLOT);
    return;
  }
  constexpr int V16 = D / 8;  // 16-byte vectors per row
  const long long src = ((long long)un.b * ws.n_kv_heads + un.g) * D;
  const long long dst = (((long long)a.layer * ws.pool_slots + loc) * ws.n_kv_heads + un.g) * D;
  for (int i = lane; i < 2 * V16; i += 32) {
    const bool isv = i >= V16;
    const int v = isv ? i - V16 : i;
    const uint4 x = reinterpret_cast<const uint4 *>(
        static_cast<const uint16_t *>(isv ? a.v_new : a.k_new) + src)[v];
    reinterpret_cast<uint4 *>(static_cast<uint16_t *>(isv ? ws.v_pool : ws.k_pool) + dst)[v] = x;
  }
  // The row must be visible to the async-proxy loads issued next.
  asm volatile("fence.proxy.async.global;" ::: "memory");
  __syncwarp();
}

// Producer, page mode: one tensor-map box per 16-token page piece and pool
// (both halves of the rows).  Lanes j and j + 4 (j < 4) both resolve piece j
// from its page id `raw` (fetched ahead) and load its K and its V; lane j
// records the piece's error bit.  A bad page id loads an in-range dummy piece
// instead (its unit is written empty), so the byte count follows from the
// tile's length alone and no warp vote is needed.
template <int D, int G>
__device__ __forceinline__ void produce_tma(const DecodeArgs &a, const Plan &pl, const Unit &un,
                                            int tile0, int raw, int stage, uint32_t kv_base,
                                            uint64_t *full, int *flag4, const CUtensorMap *tmk,
                                            const CUtensorMap *tmv, int lane) {
  using C = MCfg<D, G>;
  const pkv_workspace &ws = a.ws;
  if (lane < 8) {
    const int j = lane & 3;
    const int tok0 = tile0 + 16 * j;
    int kind = 0;
    if (tok0 < un.t1) {
      long long slot0 = slot_from_raw(ws, pl, raw, tok0, kind);  // tok0 % 16 == 0: one page
      if (kind) {
        if (lane < 4) atomicOr(ws.err, kind);
        slot0 = 0;
      }
      tma_load_4d(kv_base + stage * 2 * C::TILE + j * 2 * C::PIECE + (lane >> 2) * C::PIECE,
                  lane < 4 ? tmk : tmv, 0, a.layer * ws.pool_slots + (int)slot0, 0, un.g, full);
    }
    if (lane < 4) flag4[lane] = kind;
  }
  __syncwarp();  // the lanes' flags before the arrival that publishes the stage
  if (lane == 0)
    mbar_arrive_expect_tx(full, min(4, (un.t1 - tile0 + 15) / 16) * (uint32_t)(2 * C::PIECE));
}

// Producer, any page size / flat mode: validate the tile's index entries.
// Lane l resolves rows l and l + 32 of the tile to pool slots (-1: past the
// unit's end or a bad entry, which raises its error bit and flags the stage)
// and writes them, with the unit's KV head, for the consumer warps, which
// copy their own 16 rows each (gather_rows).
template <int D>
__device__ __forceinline__ void validate_rows(const DecodeArgs &a, const Plan &pl, const Unit &un,
                                              int tile0, const int (&raw)[2], int *srow,
                                              int *sg, int *flag4, int lane) {
  const pkv_workspace &ws = a.ws;
  int kind = 0;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int tok = tile0 + lane + 32 * h;
    srow[lane + 32 * h] = tok < un.t1 ? (int)slot_from_raw(ws, pl, raw[h], tok, kind) : -1;
  }
  const int bad = __reduce_or_sync(0xffffffffu, kind);
  if (lane < 4) flag4[lane] = lane == 0 ? bad : 0;
  if (lane == 0) {
    *sg = un.g;
    if (bad) atomicOr(ws.err, bad);
  }
}

// Consumer warp w, gather path: 16-byte cp.async copies of its own 16 rows
// (tokens 16w .. 16w + 15) of a tile's K and V into the stage, D / 8 lanes
// per row (whole 128-byte lines), zero-filled where the row has no slot.
template <int D, int G>
__device__ __forceinline__ void gather_rows(const DecodeArgs &a, const int *srow, int g,
                                            uint32_t kt, int warp, int lane) {
  using C = MCfg<D, G>;
  constexpr int CH = D / 8;     // 16-byte chunks per row
  constexpr int RPI = 32 / CH;  // rows per warp instruction
  const pkv_workspace &ws = a.ws;
  const int sub = lane / CH, ch = lane % CH;
  const long long head0 = ((long long)a.layer * ws.pool_slots * ws.n_kv_heads + g) * D + ch * 8;
  const uint16_t *kb = static_cast<const uint16_t *>(ws.k_pool) + head0;
  const uint16_t *vb = static_cast<const uint16_t *>(ws.v_pool) + head0;
  const long long slot_elems = (long long)ws.n_kv_heads * D;
  const uint32_t vt = kt + C::PIECE;
#pragma unroll
  for (int i = 0; i < 16 / RPI; ++i) {
    const int r = 16 * warp + i * RPI + sub;
    const int sl = srow[r];
    const long long e = sl >= 0 ? sl * slot_elems : 0;
    const uint32_t off = kv_off<C::HALVES>(r, ch >> 3, ch & 7);
    cp_async_16(kt + off, kb + e, sl >= 0 ? 16 : 0);
    cp_async_16(vt + off, vb + e, sl >= 0 ? 16 : 0);
  }
}

// TMA: the page-mode producer issues tensor-map boxes; else it validates
// index entries and the consumer warps issue their own cp.async gathers.
template <int D, int G, bool TMA>
__global__ void __launch_bounds__(kMThreads, 2)
    decode_mma_kernel(const __grid_constant__ DecodeArgs a, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv) {
  constexpr bool use_tma = TMA;
  using C = MCfg<D, G>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[kMStages], empty[kMStages];
  __shared__ int flags[kMStages][4];  // per stage: error bits of the tile's four pieces
  __shared__ volatile int s_ctrl[2];  // abort flag, merge ticket
  __shared__ float s_ml[kCW * 16 * 2];
  __shared__ float s_hml[16][2];  // (M, L) of each query head of the unit's group
  __shared__ int s_bad[kCW];
  __shared__ int s_pref[kMaxCompactBatch + 1];
  __shared__ int s_len[kMaxCompactBatch];
  __shared__ int s_base[kMaxCompactBatch];
  __shared__ int s_chunk[kMaxCompactBatch];
  __shared__ __align__(16) int s_idx[kLA][64];  // index entries of tiles k .. k + kLA - 1
  __shared__ int s_tmp[32];
  __shared__ int s_max_len;
  // gather path: the tile's KV head per stage, written by the producer with
  // the tile's validated slots (over its index-ring entries) before the
  // stage's full barrier; per consumer warp and stage, its tile's error bits
  __shared__ int s_sg[TMA ? 1 : kMStages];
  __shared__ int s_wbad[TMA ? 1 : kCW][TMA ? 1 : kMStages];
  uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const pkv_workspace &ws = a.ws;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Hq = ws.n_q_heads;
  volatile int *s_abort = &s_ctrl[0];
  volatile int *s_ticket = &s_ctrl[1];
  // Without PKV_FLAG_PLAN_EARLY nothing is read before the previous kernel
  // on the stream has finished.
  const bool early = (a.flags & PKV_FLAG_PLAN_EARLY) != 0;
  if (use_tma && tid == kCW * 32) {
    // fetch both descriptors while the plan is built
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmk) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmv) : "memory");
  }
  if (!early) pdl_wait();

  // The producer's lane 0 sets up the barriers while warp 0 plans; the plan's
  // block barrier publishes them before any use.
  if (tid == kCW * 32) {
    for (int s = 0; s < kMStages; ++s) {
      // TMA: one expect-tx arrival; gathers: the arrival that publishes the
      // stage's slots.  empty: the four consumer warps (gathers: each once
      // it has issued its copies of the stage's tile).
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kCW);
    }
    *s_abort = 0;
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (tid == kCW * 32) fence_barrier_init();

  Plan pl;
  pl.set_pages(ws);
  pl.batch = a.batch;
  pl.hkv = ws.n_kv_heads;
  pl.S = a.num_splits;
  const bool direct = pl.S == 1;
  const bool fused = a.fused_merge && !direct;
  // The step's plan (PKV_FLAG_USE_PLAN): every thread reads the header and
  // its share of the arrays in one round trip, and they are used only if the
  // header was written for exactly this launch; else the block plans below.
  bool planned = false;
  if ((a.flags & PKV_FLAG_USE_PLAN) && ws.work_plan && a.batch <= kMaxCompactBatch &&
      gridDim.x <= kPlanMaxGrid) {
    const int *P = ws.work_plan;
    const int apportioned = a.apportion && fused ? 1 : 0;
    int h[10];
#pragma unroll
    for (int i = 0; i < 10; ++i) h[i] = __ldcg(P + i);
    constexpr int kPer = (kMaxCompactBatch + kMThreads) / kMThreads;  // batch + 1 entries
    constexpr int nthr = kMThreads;
    int vp[kPer], vl[kPer], vb[kPer], vc[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int b = tid + j * nthr;
      if (b <= a.batch) vp[j] = __ldcg(P + kPlanPref + b);
      if (b < a.batch) {
        vl[j] = __ldcg(P + kPlanLen + b);
        vb[j] = __ldcg(P + kPlanBase + b);
        vc[j] = __ldcg(P + kPlanChunk + b);
      }
    }
    const int first =
        use_tma && tid < kLA * 4 ? __ldcg(P + kPlanFirst + blockIdx.x * kLA * 4 + tid) : -1;
    planned = h[kHMagic] == kPlanMagic && h[kHBatch] == a.batch && h[kHSplits] == pl.S &&
              h[kHGrid] == (int)gridDim.x && h[kHApportion] == apportioned &&
              h[kHTma] == (use_tma ? 1 : 0) && h[kHHkv] == pl.hkv;
    if (planned) {
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int b = tid + j * nthr;
        if (b <= a.batch) s_pref[b] = vp[j];
        if (b < a.batch) {
          s_len[b] = vl[j];
          s_base[b] = vb[j];
          s_chunk[b] = vc[j];
        }
      }
      if (use_tma && tid < kLA * 4) s_idx[tid >> 2][tid & 3] = first;
      pl.pref = s_pref;
      pl.lens = s_len;
      pl.chunks = apportioned ? s_chunk : nullptr;
      pl.chunk = h[kHChunk];
      pl.n_units = h[kHUnits];
    }
    __syncthreads();  // also publishes the barriers set up above
  }
  if (!planned) {
    if (a.batch <= kMaxCompactBatch) {
      const int budget = a.apportion && fused ? (int)gridDim.x : 0;
      const int pairs = batch_plan_compact(ws, a.batch, pl.S, budget, s_len, s_base, s_pref,
                                           s_chunk, s_tmp, &s_max_len, &pl.chunk);
      pl.pref = s_pref;
      pl.lens = s_len;
      pl.chunks = budget > 0 ? s_chunk : nullptr;
      pl.n_units = pairs * pl.hkv;
    } else {
      pl.chunk = split_chunk(batch_max_len(ws, a.batch, &s_max_len), pl.S, ws.page_size);
      pl.n_units = pl.S * pl.batch * pl.hkv;
    }
  }
  const uint32_t kv_base = smem_addr(smem + C::OFF_KV);

  // Gather path: the 64 index entries of each of the first kLA tiles are
  // fetched by the whole block at once (each thread walks its own cursor to
  // its entries' tile); the TMA path's 4 per tile are left to the producer.
  if (!use_tma) {
    Cursor<kMT> c;
    int at = -1;
    for (int e = tid; e < kLA * kMT; e += kMThreads) {
      const int tile = e / kMT, r = e - tile * kMT;
      if (at < 0) {
        c.start(ws, pl);
        at = 0;
      }
      c.advance_by(ws, pl, tile - at);
      at = tile;
      int v = -1;
      if (!c.done) {
        const Unit &u = c.it.un;
        const int tok = u.t0 + c.i * kMT + r;
        const ReqIndex ri = pl.pref ? req_index_cached(ws, s_base, u.b) : req_index(ws, u.b);
        if (tok < u.t1 && ri.ok) {
          // a 4-byte asynchronous copy: every thread's entries in flight at once
          asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(&s_idx[tile][r])),
                       "l"(index_src(ws, pl, ri, tok))
                       : "memory");
          continue;
        }
      }
      s_idx[tile][r] = v;
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
  }

  if (warp == kCW) {
    // ------------------------------------------------------- producer ----
    // pc walks the tiles to issue.  The index entries of the first kLA tiles
    // are fetched at once, lane-strided, with 4-byte cp.async copies (each
    // lane walks a copy of pc to its entry's tile); pf then runs ahead and
    // fetches later entries the same way into the ring, one commit group per
    // tile, so no register ever waits on an index load.  TMA path: entries
    // 0..3 of a ring slot are the page ids of the tile's 16-token pieces;
    // gather path: entries 0..63 are the slots / page ids of its rows,
    // replaced by the validated slots the consumer warps copy from; -1 where
    // there is none.
    Cursor<kMT> pc;
    pc.start(ws, pl);
    if (use_tma && !planned) {
      const int per = 4;
      Cursor<kMT> c = pc;
      int at = 0;
      for (int e = lane; e < kLA * per; e += 32) {
        const int tile = e / per, r = e - tile * per;
        c.advance_by(ws, pl, tile - at);
        at = tile;
        int *dst = &s_idx[tile][r];
        bool want = false;
        const int *src = nullptr;
        if (!c.done) {
          const Unit &u = c.it.un;
          const int tok = u.t0 + c.i * kMT + 16 * r;
          const ReqIndex ri = pl.pref ? req_index_cached(ws, s_base, u.b) : req_index(ws, u.b);
          want = tok < u.t1 && ri.ok;
          if (want) src = index_src(ws, pl, ri, tok);
        }
        if (want)
          asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src)
                       : "memory");
        else
          *dst = -1;
      }
    }
    Cursor<kMT> pf = pc;
    // TMA: entries are fetched kLA tiles ahead.  Gathers: the ring slot of
    // tile k holds its validated slots until every consumer warp has issued
    // tile k, which the producer knows at iteration k + kMStages (its empty
    // wait), so entries are fetched kLA - kMStages tiles ahead, into the slot
    // of tile k - kMStages.
    constexpr int kAhead = TMA ? kLA : kLA - kMStages;
    pf.advance_by(ws, pl, kAhead);
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncwarp();
    int pf_u = -1;
    ReqIndex pf_ri{0, false};
    // entries of the tile under pf into s_idx[slot], then pf moves on
    auto prefetch = [&](int slot) {
      const Unit &fu = pf.it.un;
      if (!pf.done && fu.u != pf_u) {
        pf_ri = pl.pref ? req_index_cached(ws, s_base, fu.b) : req_index(ws, fu.b);
        pf_u = fu.u;
      }
      const int tile0 = pf.done ? 0 : fu.t0 + pf.i * kMT;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int r = lane + 32 * h;
        const int tok = use_tma ? tile0 + 16 * r : tile0 + r;
        const bool want = (use_tma ? r < 4 : true) && !pf.done && tok < fu.t1 && pf_ri.ok;
        int *dst = &s_idx[slot][r];
        if (want) {
          const int *src = index_src(ws, pl, pf_ri, tok);
          asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src)
                       : "memory");
        } else {
          *dst = -1;
        }
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
      if (!pf.done) pf.advance(ws, pl);
    };
    int k = 0;
    bool aborted = false;
    bool waited = !early;
    if (waited) pdl_trigger();
    while (!pc.done) {
      const int s = k % kMStages;
      const int r = k / kMStages;
      if (r > 0 && !mbar_wait_bounded(&empty[s], (r - 1) & 1)) {
        aborted = true;
        break;
      }
      if (*s_abort) {
        aborted = true;
        break;
      }
      const Unit un = pc.it.un;
      const int tile0 = un.t0 + pc.i * kMT;
      if (!waited && a.k_new != nullptr && un.L > 0 && un.L - 1 >= tile0 &&
          un.L - 1 < min(tile0 + kMT, un.t1)) {
        pdl_wait();  // k_new comes from the previous kernel
        pdl_trigger();
        waited = true;
      }
      append_if_newest<D>(a, un, tile0, lane);
      // tile k's entries: at most kAhead - 1 newer groups pend
      asm volatile("cp.async.wait_group %0;" ::"n"(kAhead - 1) : "memory");
      const int slot = k % kLA;
      // TMA: lanes j and j + 4 both need piece j's page id
      const int cur[2] = {s_idx[slot][use_tma ? (lane & 3) : lane], s_idx[slot][lane + 32]};
      __syncwarp();
      if (k == 0 && (a.flags & PKV_FLAG_TEST_SKIP_FIRST_TILE)) {
        // test hook: the stage is never armed, the consumers' wait runs out
      } else if (use_tma) {
        produce_tma<D, G>(a, pl, un, tile0, cur[0], s, kv_base, &full[s], flags[s], &tmk, &tmv,
                          lane);
      } else if constexpr (!TMA) {
        validate_rows<D>(a, pl, un, tile0, cur, s_idx[slot], &s_sg[s], flags[s], lane);
        __syncwarp();  // every lane's slots before the arrival that publishes them
        if (lane == 0) mbar_arrive(&full[s]);
      }
      pc.advance(ws, pl);
      prefetch((k + kAhead) % kLA);  // TMA: the slot just read
      ++k;
    }
    if (aborted) {
      if (lane == 0) {
        *s_abort = 1;
        atomicOr(ws.err, PKV_DEVERR_TIMEOUT);
      }
      // Drain: the last (up to kMStages) issued tiles may still be landing.
      for (int kk = max(0, k - kMStages); kk < k; ++kk)
        mbar_wait_bounded(&full[kk % kMStages], (kk / kMStages) & 1);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");  // index copies still in flight
    return;
  }

  // ---------------------------------------------------------- consumers ----
  const int grp = lane >> 2, tig = lane & 3;
  // This lane's B/C columns are heads 2*tig + e (+ 8*n for the n-th head tile).
  const float qk_scale = a.scale * kLog2e;
  float *red = reinterpret_cast<float *>(smem + C::OFF_RED);
  // ldmatrix lane addressing in the swizzled layout: matrix mi = lane / 8,
  // row rr = lane % 8 of that matrix.
  const int mi = lane >> 3, rr = lane & 7;
  const int rowK = 16 * warp + (mi & 1) * 8 + rr;   // K as A: tokens 0-7 / 8-15 by mi % 2
  const int rowV = 16 * warp + (mi >> 1) * 8 + rr;  // V^T as A: tokens by mi / 2

  // q and every output belong to the current stream order: wait here, then
  // let the next kernel on the stream be scheduled.
  if (early) pdl_wait();
  pdl_trigger();
  if (pl.pref && (direct || fused)) {
    // Requests with no usable token have no unit: zero their outputs here.
    for (int b = blockIdx.x; b < a.batch; b += gridDim.x) {
      if (s_pref[b + 1] != s_pref[b]) continue;
      for (int i = tid; i < Hq * D; i += kCW * 32) {
        const long long o = (long long)b * Hq * D + i;
        if (a.flags & PKV_FLAG_OUT_F32) static_cast<float *>(ws.out)[o] = 0.f;
        else static_cast<uint16_t *>(ws.out)[o] = 0;
      }
      if ((a.flags & PKV_FLAG_WRITE_LSE) && ws.lse)
        for (int h = tid; h < Hq; h += kCW * 32) ws.lse[(long long)b * Hq + h] = -INFINITY;
    }
  }

  // Gather path: each consumer warp copies its own rows of tile t two tiles
  // ahead (at tile t - 2): it waits for the producer to publish the stage's
  // slots, issues its copies as one cp.async group and releases the slots;
  // before computing a tile it waits for its own group.  The stage it fills
  // held tile t - 3, which this warp has finished.
  int tiles_total = 0;
  auto issue = [&](int t) {
    const int st = t % kMStages;
    bool ok = false;
    if (!*s_abort) {
      ok = mbar_wait_bounded(&full[st], (t / kMStages) & 1);
      if (!ok && lane == 0) {
        *s_abort = 1;
        atomicOr(ws.err, PKV_DEVERR_TIMEOUT);
      }
    }
    if (ok) {
      gather_rows<D, G>(a, s_idx[t % kLA], s_sg[st], kv_base + st * 2 * C::TILE, warp, lane);
      if (lane == 0) s_wbad[warp][st] = flags[st][0] | flags[st][1] | flags[st][2] | flags[st][3];
    } else if (lane == 0) {
      s_wbad[warp][st] = PKV_DEVERR_TIMEOUT;
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    __syncwarp();  // every lane has read the stage's slots
    if (lane == 0) mbar_arrive(&empty[st]);
  };
  if constexpr (!TMA) {
    UnitIter u2;
    u2.first(ws, pl);
    for (; !u2.done; u2.next(ws, pl))
      if (u2.un.t0 < u2.un.t1) tiles_total += (u2.un.t1 - u2.un.t0 + kMT - 1) / kMT;
    for (int t = 0; t < 2 && t < tiles_total; ++t) issue(t);
  }

  int k = 0;
  UnitIter ui;
  ui.first(ws, pl);
  for (; !ui.done; ui.next(ws, pl)) {
    const Unit un = ui.un;
    const int hq0 = un.g * G;
    const int n_b = un.n;
    if (un.t0 >= un.t1) {  // dense enumeration only
      const int ct = tid;  // consumer thread 0..127
      if (direct || fused) {
        if (un.c == 0) {  // a request with no tokens: zero output
          for (int i = ct; i < G * D; i += kCW * 32) {
            const long long o = ((long long)un.b * Hq + hq0) * D + i;
            if (a.flags & PKV_FLAG_OUT_F32) static_cast<float *>(ws.out)[o] = 0.f;
            else static_cast<uint16_t *>(ws.out)[o] = 0;
          }
          if ((a.flags & PKV_FLAG_WRITE_LSE) && ws.lse && ct < G)
            ws.lse[(long long)un.b * Hq + hq0 + ct] = -INFINITY;
        }
      } else if (ct < G) {
        const long long o = (((long long)un.b * Hq + hq0 + ct) * pl.S + un.c) * 2;
        ws.ml_part[o] = -INFINITY;
        ws.ml_part[o + 1] = 0.f;
      }
      continue;
    }
    const int ntiles = (un.t1 - un.t0 + kMT - 1) / kMT;

    // Q^T as the B operand: b0 = Q[h][d0 + 2 tig ..], b1 = Q[h][d0 + 8 + 2 tig ..]
    // for h = grp + 8 n (heads >= G are zero).
    uint32_t qb[C::NH][C::KSTEPS][2];
    {
      const uint32_t *q32 = static_cast<const uint32_t *>(a.q);
#pragma unroll
      for (int n = 0; n < C::NH; ++n) {
        const int h = grp + 8 * n;
        const long long row = ((long long)un.b * Hq + hq0 + h) * (D / 2);
#pragma unroll
        for (int ks = 0; ks < C::KSTEPS; ++ks) {
          qb[n][ks][0] = h < G ? q32[row + ks * 8 + tig] : 0u;
          qb[n][ks][1] = h < G ? q32[row + ks * 8 + tig + 4] : 0u;
        }
      }
    }
    // O^T accumulators: acc[n][mt] = O[h = 8n + 2 tig + {0,1}][d = 16 mt + grp (+8)]
    float acc[C::NH][C::MT][4];
#pragma unroll
    for (int n = 0; n < C::NH; ++n)
#pragma unroll
      for (int mt = 0; mt < C::MT; ++mt) acc[n][mt][0] = acc[n][mt][1] = acc[n][mt][2] = acc[n][mt][3] = 0.f;
    float m_run[C::NH][2], l_run[C::NH][2];
#pragma unroll
    for (int n = 0; n < C::NH; ++n) {
      m_run[n][0] = m_run[n][1] = -INFINITY;
      l_run[n][0] = l_run[n][1] = 0.f;
    }
    int bad = 0;

    for (int it = 0; it < ntiles; ++it, ++k) {
      const int s = k % kMStages;
      bool ok = false;
      if constexpr (TMA) {
        if (!*s_abort) {
          ok = mbar_wait_bounded(&full[s], (k / kMStages) & 1);
          if (!ok && lane == 0) {
            *s_abort = 1;
            atomicOr(ws.err, PKV_DEVERR_TIMEOUT);
          }
        }
      } else {
        if (k + 2 < tiles_total) issue(k + 2);
        // this warp's copies of tile k: the groups of tiles k+1, k+2 may pend
        const int newer = min(2, tiles_total - 1 - k);
        if (newer >= 2) asm volatile("cp.async.wait_group 2;" ::: "memory");
        else if (newer == 1) asm volatile("cp.async.wait_group 1;" ::: "memory");
        else asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncwarp();  // the lanes' rows visible to the whole warp
        ok = s_wbad[warp][s] != PKV_DEVERR_TIMEOUT;
      }
      const int nv = min(16, un.t1 - (un.t0 + it * kMT) - 16 * warp);  // my valid tokens
      if (!ok) {
        bad = 1;
      } else {
        if constexpr (TMA) bad |= flags[s][0] | flags[s][1] | flags[s][2] | flags[s][3];
        else bad |= s_wbad[warp][s];
        if (nv > 0) {
          const uint32_t kt = kv_base + s * 2 * C::TILE;  // K then V per 16-token piece
          const uint32_t vt = kt + C::PIECE;
          // ---- S^T = K Q^T: rows = tokens grp / grp + 8, cols = heads ----
          // two independent accumulation chains (even / odd k-steps)
          float sc[C::NH][4], sc2[C::NH][4];
#pragma unroll
          for (int n = 0; n < C::NH; ++n)
#pragma unroll
            for (int i = 0; i < 4; ++i) sc[n][i] = sc2[n][i] = 0.f;
#pragma unroll
          for (int ks = 0; ks < C::KSTEPS; ++ks) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(kt + kv_off<C::HALVES>(rowK, ks >> 2, (ks & 3) * 2 + (mi >> 1)), a0, a1, a2,
                    a3);
#pragma unroll
            for (int n = 0; n < C::NH; ++n)
              mma_bf16_16816((ks & 1) ? sc2[n] : sc[n], a0, a1, a2, a3, qb[n][ks][0], qb[n][ks][1]);
          }
#pragma unroll
          for (int n = 0; n < C::NH; ++n)
#pragma unroll
            for (int i = 0; i < 4; ++i) sc[n][i] += sc2[n][i];
          if (nv < 16) {
            // Rows past the end of this warp's piece may hold anything the
            // pool held (even NaN bit patterns); P is 0 there, so clear them.
            for (int i = lane; i < (16 - nv) * 16; i += 32) {
              const int r = 16 * warp + nv + (i >> 4), c8 = i & 15;
              if (c8 < D / 8)
                asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(
                                 vt + kv_off<C::HALVES>(r, c8 >> 3, c8 & 7)),
                             "r"(0u)
                             : "memory");
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
          }
          // ---- online softmax over the tokens, per head (log2 units) ----
          const bool v0 = grp < nv, v1 = grp + 8 < nv;
          uint32_t bh[C::NH][2], bl[C::NH][2];  // P^T as B: tokens 0-7 / 8-15
#pragma unroll
          for (int n = 0; n < C::NH; ++n) {
            float al[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float s0 = v0 ? sc[n][e] * qk_scale : -INFINITY;
              const float s1 = v1 ? sc[n][2 + e] * qk_scale : -INFINITY;
              float t = fmaxf(s0, s1);
              t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, 4));
              t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, 8));
              t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, 16));
              const float mn = fmaxf(m_run[n][e], t);
              al[e] = exp2f(m_run[n][e] - mn);
              m_run[n][e] = mn;
              const float p0 = exp2f(s0 - mn), p1 = exp2f(s1 - mn);
              l_run[n][e] = l_run[n][e] * al[e] + p0 + p1;
              sc[n][e] = p0;
              sc[n][2 + e] = p1;
            }
#pragma unroll
            for (int mt = 0; mt < C::MT; ++mt) {
              acc[n][mt][0] *= al[0];
              acc[n][mt][1] *= al[1];
              acc[n][mt][2] *= al[0];
              acc[n][mt][3] *= al[1];
            }
#pragma unroll
            for (int hlf = 0; hlf < 2; ++hlf) {
              const float x = sc[n][2 * hlf], y = sc[n][2 * hlf + 1];
              const uint32_t hi = pack_bf16x2(x, y);
              const uint32_t lo = pack_bf16x2(x - bf16lo(hi), y - bf16hi(hi));
              bh[n][hlf] = movmatrix_t(hi);
              bl[n][hlf] = movmatrix_t(lo);
            }
          }
          // ---- O^T += V^T P^T: 16 head_dim rows per mma ----
#pragma unroll
          for (int mt = 0; mt < C::MT; ++mt) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4_t(vt + kv_off<C::HALVES>(rowV, mt >> 2, (mt & 3) * 2 + (mi & 1)), a0, a1, a2,
                      a3);
#pragma unroll
            for (int n = 0; n < C::NH; ++n) {
              mma_bf16_16816(acc[n][mt], a0, a1, a2, a3, bh[n][0], bh[n][1]);
              mma_bf16_16816(acc[n][mt], a0, a1, a2, a3, bl[n][0], bl[n][1]);
            }
          }
        }
      }
      __syncwarp();
      if (TMA && lane == 0) mbar_arrive(&empty[s]);
    }

    // ---- merge the four warps' states ----
#pragma unroll
    for (int n = 0; n < C::NH; ++n)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float l = l_run[n][e];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        l_run[n][e] = l;
        if (grp == 0) {
          const int h = 8 * n + 2 * tig + e;
          s_ml[(warp * 16 + h) * 2] = m_run[n][e];
          s_ml[(warp * 16 + h) * 2 + 1] = l;
        }
      }
    if (lane == 0) s_bad[warp] = bad;
    named_sync(1, kCW * 32);
#pragma unroll
    for (int n = 0; n < C::NH; ++n)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int h = 8 * n + 2 * tig + e;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kCW; ++w) M = fmaxf(M, s_ml[(w * 16 + h) * 2]);
        float L = 0.f;
#pragma unroll
        for (int w = 0; w < kCW; ++w) {
          const float mw = s_ml[(w * 16 + h) * 2];
          L += mw == -INFINITY ? 0.f : exp2f(mw - M) * s_ml[(w * 16 + h) * 2 + 1];
        }
        if (warp == 0 && grp == 0 && h < G) {  // lanes 0-3 of warp 0 hold every head once
          s_hml[h][0] = M;
          s_hml[h][1] = L;
        }
        const float f = m_run[n][e] == -INFINITY ? 0.f : exp2f(m_run[n][e] - M);
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt) {
          acc[n][mt][e] *= f;
          acc[n][mt][2 + e] *= f;
        }
      }
    const int unit_bad = s_bad[0] | s_bad[1] | s_bad[2] | s_bad[3];
    // tree over warps through two [G][RSTRIDE] buffers
    auto store = [&](int buf) {
#pragma unroll
      for (int n = 0; n < C::NH; ++n)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int h = 8 * n + 2 * tig + e;
          if (h >= G) continue;
          float *rowp = red + (buf * G + h) * C::RSTRIDE;
#pragma unroll
          for (int mt = 0; mt < C::MT; ++mt) {
            rowp[16 * mt + grp] = acc[n][mt][e];
            rowp[16 * mt + grp + 8] = acc[n][mt][2 + e];
          }
        }
    };
    auto add = [&](int buf) {
#pragma unroll
      for (int n = 0; n < C::NH; ++n)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int h = 8 * n + 2 * tig + e;
          if (h >= G) continue;
          const float *rowp = red + (buf * G + h) * C::RSTRIDE;
#pragma unroll
          for (int mt = 0; mt < C::MT; ++mt) {
            acc[n][mt][e] += rowp[16 * mt + grp];
            acc[n][mt][2 + e] += rowp[16 * mt + grp + 8];
          }
        }
    };
    // (w0 + w2) and (w1 + w3) land in the two buffers; every consumer thread
    // then writes four consecutive elements of their sum (coalesced).
    if (warp >= 2) store(warp - 2);
    named_sync(1, kCW * 32);
    if (warp < 2) {
      add(warp);
      store(warp);
    }
    named_sync(1, kCW * 32);

    // ---- write: final row, or a partial (and maybe merge them all) ----
    const bool final_out = direct || (fused && n_b == 1);
#pragma unroll
    for (int i = tid * 4; i < G * D; i += kCW * 32 * 4) {
      const int h = i / D, d = i - h * D;
      const float L = s_hml[h][1];
      const bool empty_out = unit_bad || !(L > 0.f);
      const float inv = empty_out ? 0.f : 1.f / L;
      const float4 x0 = *reinterpret_cast<const float4 *>(red + h * C::RSTRIDE + d);
      const float4 x1 = *reinterpret_cast<const float4 *>(red + (G + h) * C::RSTRIDE + d);
      // an empty or failed unit is written as zeros whatever its tiles held
      // (a bad page's dummy piece may hold NaN bit patterns)
      const float4 x = empty_out ? make_float4(0.f, 0.f, 0.f, 0.f)
                                 : make_float4((x0.x + x1.x) * inv, (x0.y + x1.y) * inv,
                                               (x0.z + x1.z) * inv, (x0.w + x1.w) * inv);
      const long long qrow = (long long)un.b * Hq + hq0 + h;
      if (final_out) {
        if (a.flags & PKV_FLAG_OUT_F32) {
          *reinterpret_cast<float4 *>(static_cast<float *>(ws.out) + qrow * D + d) = x;
        } else {
          uint2 pk;
          pk.x = f32_to_bf16_bits(x.x) | (f32_to_bf16_bits(x.y) << 16);
          pk.y = f32_to_bf16_bits(x.z) | (f32_to_bf16_bits(x.w) << 16);
          *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(ws.out) + qrow * D + d) = pk;
        }
      } else {
        *reinterpret_cast<float4 *>(ws.o_part + (qrow * pl.S + un.c) * D + d) = x;
      }
    }
    if (tid < G) {
      const float M = s_hml[tid][0], L = s_hml[tid][1];
      const bool empty_out = unit_bad || !(L > 0.f);
      const long long qrow = (long long)un.b * Hq + hq0 + tid;
      if (final_out) {
        if ((a.flags & PKV_FLAG_WRITE_LSE) && ws.lse)
          ws.lse[qrow] = empty_out ? -INFINITY : M * kLn2 + logf(L);
      } else {
        const long long o = (qrow * pl.S + un.c) * 2;
        ws.ml_part[o] = empty_out ? -INFINITY : M * kLn2;
        ws.ml_part[o + 1] = empty_out ? 0.f : L;
      }
    }
    if (fused && !final_out) {
      named_sync(1, kCW * 32);
      if (tid == 0) {
        // the block's partial (ordered by the barrier) is released with the
        // ticket; the last taker acquires every other block's
        int *ctr = ws.split_counters + (long long)un.b * ws.n_kv_heads + un.g;
        const int old = atomic_add_acq_rel_gpu(ctr, 1);
        const int last = old == n_b - 1;
        if (last) *ctr = 0;  // ready for the next launch
        *s_ticket = last;
      }
      named_sync(1, kCW * 32);
      if (*s_ticket) {
        // warp w merges query heads w, w + 4, ... of the group
        constexpr int RPW = G >= kCW ? G / kCW : 1;
        if (warp < G)
          merge_rows_batched<D, RPW>(ws, (long long)un.b * Hq + hq0 + warp, kCW, pl.S, n_b,
                                     a.flags, lane);
      }
    }
    named_sync(1, kCW * 32);  // s_ml, red and the ticket are reused by the next unit
  }
  if constexpr (!TMA) asm volatile("cp.async.wait_all;" ::: "memory");  // after an abort
}

using TmapEncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

TmapEncodeFn tmap_encoder() {
  static TmapEncodeFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<TmapEncodeFn>(p);
  }
  return fn;
}

// 4-D view of a pool [NL * pool_slots, Hkv, D] as (64 columns, slot, 64-column
// half, KV head), strides 2 B, Hkv * D * 2, 128, D * 2: a box of 64 x 16 x
// halves x 1 lands in shared memory as [half][slot][64 columns], one page
// piece of one head with both halves of its rows.  Every element a box can
// address lies inside the pool.  (One map over both pools, with their distance
// as a fifth stride, halves the copies per tile but ran the 65536-token single
// request ~1.5x slower.)
bool encode_pool_map(CUtensorMap *m, void *base, const pkv_workspace &ws) {
  TmapEncodeFn enc = tmap_encoder();
  if (!enc) return false;
  const cuuint64_t D = (cuuint64_t)ws.head_dim, H = (cuuint64_t)ws.n_kv_heads;
  const cuuint64_t dims[4] = {64, (cuuint64_t)ws.n_layers * (cuuint64_t)ws.pool_slots, D / 64, H};
  const cuuint64_t strides[3] = {H * D * 2, 128, D * 2};
  const cuuint32_t box[4] = {64, 16, (cuuint32_t)(D / 64), 1};
  const cuuint32_t elem[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box, elem,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Launch shape of the tensor-core decode kernel for a call: resident-block
// grid, whether its splits are apportioned, and whether TMA boxes apply (the
// tensor maps still have to encode).  The step's plan is made for the same.
struct MmaShape {
  int grid, apportion, tma;
};

template <int D, int G>
cudaError_t mma_shape(const DecodeArgs &a, MmaShape *sh) {
  using C = MCfg<D, G>;
  static int occ_cache[64] = {0};
  static int sms_cache[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int di = dev & 63;
  if (occ_cache[di] == 0) {
    // both producer paths: a launch may fall back from TMA to the gathers
    auto kt = decode_mma_kernel<D, G, true>;
    auto kg = decode_mma_kernel<D, G, false>;
    e = cudaFuncSetAttribute(kt, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kg, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    int occ = 0, occ_g = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kt, kMThreads, C::SMEM);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_g, kg, kMThreads, C::SMEM);
    if (e != cudaSuccess) return e;
    occ = occ < occ_g ? occ : occ_g;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    sms_cache[di] = sms;
    occ_cache[di] = occ > 0 ? occ : 1;
  }
  const pkv_workspace &ws = a.ws;
  const long long units = (long long)a.num_splits * a.batch * ws.n_kv_heads;
  const long long cap = (long long)sms_cache[di] * occ_cache[di];
  sh->grid = (int)(units < cap ? units : cap);
  // Apportioned splits need the compact plan, and the summed lengths must
  // fit in an int.
  sh->apportion = a.fused_merge && a.num_splits > 1 && a.batch <= kMaxCompactBatch &&
                  !(a.flags & PKV_FLAG_FIXED_CHUNK) &&
                  (long long)a.batch * ws.max_pages_per_req * ws.page_size < 0x7fffffffll;
  sh->tma = ws.index_mode == PKV_IDX_PAGE_TABLE && ws.page_size % 16 == 0 &&
            (long long)ws.n_layers * ws.pool_slots < 0x7fffffffll &&
            !(a.flags & PKV_FLAG_FORCE_GATHER);
  return cudaSuccess;
}

template <int D, int G>
cudaError_t launch_mma_one(const DecodeArgs &a, cudaStream_t st) {
  using C = MCfg<D, G>;
  MmaShape sh;
  cudaError_t e = mma_shape<D, G>(a, &sh);
  if (e != cudaSuccess) return e;
  if (sh.grid <= 0) return cudaSuccess;
  CUtensorMap tmk, tmv;
  memset(&tmk, 0, sizeof(tmk));
  memset(&tmv, 0, sizeof(tmv));
  const pkv_workspace &ws = a.ws;
  int use_tma = sh.tma;
  if (use_tma)
    use_tma = encode_pool_map(&tmk, ws.k_pool, ws) && encode_pool_map(&tmv, ws.v_pool, ws);
  DecodeArgs args = a;
  args.apportion = sh.apportion;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sh.grid);
  cfg.blockDim = dim3(kMThreads);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (use_tma) return cudaLaunchKernelEx(&cfg, decode_mma_kernel<D, G, true>, args, tmk, tmv);
  return cudaLaunchKernelEx(&cfg, decode_mma_kernel<D, G, false>, args, tmk, tmv);
}

// The step's plan (see pkv_plan_step): the compact plan every decode block
// would derive, and the TMA page ids of every block's first kPlanTiles tiles
// (one thread per (block, tile)).  Block 0 writes the header and the arrays.
constexpr int kPlanThreads = 256;

__global__ void __launch_bounds__(kPlanThreads)
    plan_kernel(const __grid_constant__ pkv_workspace ws, int batch, int S, int grid,
                int apportion, int tma) {
  __shared__ int s_len[kMaxCompactBatch], s_base[kMaxCompactBatch], s_chunk[kMaxCompactBatch];
  __shared__ int s_pref[kMaxCompactBatch + 1];
  __shared__ int s_tmp[32];
  __shared__ int s_max;
  Plan pl;
  pl.set_pages(ws);
  pl.batch = batch;
  pl.hkv = ws.n_kv_heads;
  pl.S = S;
  const int budget = apportion ? grid : 0;
  const int pairs =
      batch_plan_compact(ws, batch, S, budget, s_len, s_base, s_pref, s_chunk, s_tmp, &s_max,
                         &pl.chunk);
  pl.pref = s_pref;
  pl.lens = s_len;
  pl.chunks = budget > 0 ? s_chunk : nullptr;
  pl.n_units = pairs * pl.hkv;
  int *P = ws.work_plan;
  const int tid = threadIdx.x;
  if (tma) {
    for (int item = blockIdx.x * blockDim.x + tid; item < grid * kPlanTiles;
         item += gridDim.x * blockDim.x) {
      const int blk = item / kPlanTiles, t = item - blk * kPlanTiles;
      Cursor<kMT> c;
      c.start(ws, pl, blk, grid);
      c.advance_by(ws, pl, t);
      int v[4] = {-1, -1, -1, -1};
      if (!c.done) {
        const Unit &u = c.it.un;
        const ReqIndex ri = req_index_cached(ws, s_base, u.b);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int tok = u.t0 + c.i * kMT + 16 * r;
          if (tok < u.t1 && ri.ok) v[r] = *index_src(ws, pl, ri, tok);
        }
      }
      *reinterpret_cast<int4 *>(P + kPlanFirst + item * 4) = make_int4(v[0], v[1], v[2], v[3]);
    }
  }
  if (blockIdx.x == 0) {
    for (int b = tid; b < batch; b += blockDim.x) {
      P[kPlanPref + b] = s_pref[b];
      P[kPlanLen + b] = s_len[b];
      P[kPlanBase + b] = s_base[b];
      P[kPlanChunk + b] = budget > 0 ? s_chunk[b] : 0;
    }
    if (tid == 0) {
      P[kPlanPref + batch] = s_pref[batch];
      P[kHBatch] = batch;
      P[kHSplits] = S;
      P[kHGrid] = grid;
      P[kHUnits] = pl.n_units;
      P[kHChunk] = pl.chunk;
      P[kHMaxLen] = s_max;
      P[kHApportion] = budget > 0;
      P[kHTma] = tma;
      P[kHHkv] = pl.hkv;
      P[kHMagic] = kPlanMagic;
    }
  }
}

template <int D, int G>
cudaError_t launch_plan_one(const DecodeArgs &a, cudaStream_t st) {
  MmaShape sh;
  cudaError_t e = mma_shape<D, G>(a, &sh);
  if (e != cudaSuccess) return e;
  if (sh.grid <= 0 || sh.grid > kPlanMaxGrid || a.batch > kMaxCompactBatch) return cudaSuccess;
  const int items = sh.tma ? sh.grid * kPlanTiles : 1;
  const int blocks = (items + kPlanThreads - 1) / kPlanThreads;
  plan_kernel<<<blocks, kPlanThreads, 0, st>>>(a.ws, a.batch, a.num_splits, sh.grid,
                                                sh.apportion, sh.tma);
  return cudaGetLastError();
}

}  // namespace

bool decode_mma_supported(int head_dim, int group) {
  return (head_dim == 64 || head_dim == 128) &&
         (group == 1 || group == 2 || group == 4 || group == 8 || group == 16);
}

size_t plan_bytes() { return (size_t)kPlanInts * 4; }

cudaError_t launch_plan(const DecodeArgs &a, cudaStream_t st) {
  const int D = a.ws.head_dim, G = a.ws.n_q_heads / a.ws.n_kv_heads;
#define PKV_PLAN_CASE(DD, GG) \
  if (D == DD && G == GG) return launch_plan_one<DD, GG>(a, st);
  PKV_PLAN_CASE(128, 1) PKV_PLAN_CASE(128, 2) PKV_PLAN_CASE(128, 4) PKV_PLAN_CASE(128, 8)
  PKV_PLAN_CASE(128, 16) PKV_PLAN_CASE(64, 1) PKV_PLAN_CASE(64, 2) PKV_PLAN_CASE(64, 4)
  PKV_PLAN_CASE(64, 8) PKV_PLAN_CASE(64, 16)
#undef PKV_PLAN_CASE
  return cudaErrorNotSupported;
}

cudaError_t launch_decode_mma(const DecodeArgs &a, cudaStream_t st) {
  const int D = a.ws.head_dim, G = a.ws.n_q_heads / a.ws.n_kv_heads;
#define PKV_MMA_CASE(DD, GG) \
  if (D == DD && G == GG) return launch_mma_one<DD, GG>(a, st);
  PKV_MMA_CASE(128, 1) PKV_MMA_CASE(128, 2) PKV_MMA_CASE(128, 4) PKV_MMA_CASE(128, 8)
  PKV_MMA_CASE(128, 16) PKV_MMA_CASE(64, 1) PKV_MMA_CASE(64, 2) PKV_MMA_CASE(64, 4)
  PKV_MMA_CASE(64, 8) PKV_MMA_CASE(64, 16)
#undef PKV_MMA_CASE
  return cudaErrorNotSupported;
}

}  // namespace pkv
