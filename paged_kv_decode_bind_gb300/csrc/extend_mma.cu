// Paged extend (prefill) attention on the tensor cores, and the append of the
// new tokens' K/V.  The per-request query offsets qo_indptr are the ones the
// engine keeps in its workspace for the prefill step (workspace.py page,
// bullet 19).  Request b holds L_b tokens in the pool, the last n_b of them
// new (qo_indptr[b + 1] - qo_indptr[b]); new token i sits at position
// L_b - n_b + i and attends causally to tokens 0 .. L_b - n_b + i
// (PKV_FLAG_EXTEND_FULL: every row attends all L_b tokens, as a batch's
// decode queries over a prefix their requests share).
//
// Math.  A block computes 64 query rows of one (request, KV head): rows are
// (new token, query head of the group) pairs, 64 / G tokens x G heads, so a
// key tile is read once for the whole group.  Each of four consumer warps
// owns 16 rows: S = Q K^T with warp-level bf16 mma.m16n8k16 (query rows on
// the 16-row side, 8 keys per n-tile, fp32 accumulation), the causal mask
// and an online softmax in fp32 (exp2), then O += P V with P rounded to bf16
// (8 mantissa bits: each weight's rounding error is at most 2^-9 of it, far
// inside the 1e-2 output tolerance; splits agree within 2e-3).
// The accumulator fragment of S is the A fragment of P as it stands, so no
// transpose is needed.
//
// Pipeline.  One producer warp fills a 3-stage ring (full / empty
// mbarriers) with each 64-key tile's K and V, laid out per 16-token piece as
// [64-column half][16 rows][128 B] with the 128-byte swizzle, a piece's K
// then its V.  Page sizes that are multiples of 16 use one tensor-map box per
// piece and pool (the copy engine writes shared memory directly, leaving the
// load/store pipe to the consumers' ldmatrix); other page sizes and flat
// indices use 16-byte cp.async gathers.  The next tile's index entries load
// while the current tile's copies are issued.  Every wait is bounded (~1 s)
// and raises PKV_DEVERR_TIMEOUT.
//
// Work.  Units are (query block j, split c, request, KV head), visited in
// order of decreasing j so that the longest causal ranges start first; a
// persistent grid strides over them.  With S > 1 splits each split writes
// its rows' normalised partials and (m, l) to the workspace's o_part /
// ml_part and extend_merge_kernel combines them.  Invalid requests (n_b < 0,
// n_b > L_b in the causal mode, n_b > max_qo_len, rows past qo_indptr[batch],
// L_b out of range, or, when the workspace's partials or lse are written,
// rows past the batch * max_qo_len it holds) raise PKV_DEVERR_LEN and get no
// output rows; a bad page id or flat slot
// raises its bit and writes the unit's rows as zeros.  merge_lse_kernel
// combines two results over disjoint keys of the same rows (a shared
// prefix's and each request's own suffix's).
#include <climits>

#include <cuda.h>

#include <cstring>
#include <utility>

#include "extend_common.cuh"
#include "merge.cuh"

namespace pkv {

cudaError_t launch_extend(const pkv_workspace &ws, int batch, int layer, const int *qo_indptr,
                          int max_qo_len, const void *q, void *out, float scale, int num_splits,
                          int flags, cudaStream_t st);
cudaError_t launch_extend_append(const pkv_workspace &ws, int batch, int layer,
                                 const int *qo_indptr, int max_qo_len, const void *k_new,
                                 const void *v_new, cudaStream_t st);
bool extend_supported(int head_dim, int group);
cudaError_t launch_merge_lse(int n_rows, int head_dim, const float *o_a, const float *lse_a,
                             const float *o_b, const float *lse_b, void *out, float *lse_out,
                             int flags, cudaStream_t st);

namespace {

constexpr int kXW = 4;                  // consumer warps
constexpr int kXThreads = (kXW + 1) * 32;
constexpr int kXRows = 16 * kXW;        // query rows per block
constexpr int kXStages = 3;

template <int D>
struct XCfg {
  static constexpr int HALVES = D / 64;
  static constexpr int PIECE = 16 * HALVES * 128;  // K (or V) of a 16-token piece
  static constexpr int TILE = (kXT / 16) * PIECE;  // K (or V) of a tile
  static constexpr int STAGE = 2 * TILE;
  static constexpr int KSTEPS = D / 16;
  static constexpr int ND = D / 8;              // 8-column output tiles
  static constexpr int SMEM = kXStages * STAGE + 1024;  // + alignment slack
  static_assert(D % 64 == 0 && KSTEPS % 2 == 0, "whole swizzled halves, paired k-steps");
};

// Byte offset of 16-byte chunk ch (0 .. D/8 - 1) of key row t from the
// stage's K base (the V base is one piece further): piece t / 16, then
// [half][row][128 B] with chunk c of row r at c ^ (r & 7).
template <int D>
__device__ __forceinline__ uint32_t xoff(int t, int ch) {
  return (uint32_t)((t >> 4) * 2 * XCfg<D>::PIECE + (((ch >> 3) * 16 + (t & 15)) * 128) +
                    (((ch & 7) ^ (t & 7)) << 4));
}

__device__ __forceinline__ void xtma4(uint32_t dst, const CUtensorMap *tm, int c1, int c3,
                                      uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], "
      "[%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(0), "r"(c1), "r"(0), "r"(c3), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void xcp16(uint32_t dst, const void *src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}

// TMA: the page-piece boxes (P % 16 == 0); else the cp.async gathers.
template <int D, int G, bool TMA>
__global__ void __launch_bounds__(kXThreads, 2)
    extend_mma_kernel(const __grid_constant__ XArgs a, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv) {
  // With programmatic dependent launch everything read here may come from
  // the previous kernel on the stream: wait for it (a no-op for a plain
  // launch), then let the next kernel be scheduled.
  pdl_wait();
  pdl_trigger();
  using C = XCfg<D>;
  constexpr int TQ = kXRows / G;  // new tokens per block
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[kXStages], empty[kXStages];
  __shared__ int flags[kXStages];
  __shared__ int s_slot[kXStages][kXT];
  __shared__ volatile int s_abort;
  uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const pkv_workspace &ws = a.ws;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Hq = ws.n_q_heads;
  const int jmax = (a.max_qo_len + TQ - 1) / TQ;
  const int units = jmax * a.S * a.batch * ws.n_kv_heads;
  if (tid == kXW * 32) {
    if (TMA) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(&tmk) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(&tmv) : "memory");
    }
    for (int s = 0; s < kXStages; ++s) {
      // TMA: one expect-tx arrival; gathers: 32 copy-completion arrivals +
      // the flag writer's
      mbar_init(&full[s], TMA ? 1 : 33);
      mbar_init(&empty[s], kXW);
    }
    s_abort = 0;
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (tid == kXW * 32) fence_barrier_init();
  __syncthreads();
  const uint32_t ring = smem_addr(smem);

  if (warp == kXW) {
    // ------------------------------------------------------- producer ----
    Plan pl;
    pl.set_pages(ws);
    constexpr int CH = D / 8;     // 16-byte chunks per row
    constexpr int RPI = 32 / CH;  // rows per warp instruction
    const int sub = lane / CH, ch = lane % CH;
    const long long slot_elems = (long long)ws.n_kv_heads * D;
    int k = 0;
    bool aborted = false;
    for (int u = blockIdx.x; u < units && !aborted; u += gridDim.x) {
      const XUnit x = xunit(a, u, TQ, jmax);
      if (!x.live) continue;
      long long base = 0;
      bool row_ok = true;
      if (ws.index_mode == PKV_IDX_FLAT) {
        base = ws.kv_indptr[x.b];
      } else {
        const int row = ws.req_pool_indices[x.b];
        row_ok = row >= 0 && row < ws.max_reqs;
        base = row_ok ? (long long)row * ws.max_pages_per_req : 0;
      }
      const int *idx = ws.index_mode == PKV_IDX_FLAT ? ws.kv_indices : ws.page_table;
      auto raw_at = [&](int t) {
        if (t >= x.k1 || !row_ok) return -1;
        return idx[base + (ws.index_mode == PKV_IDX_FLAT ? t : pl.page_of(t))];
      };
      const long long head0 = ((long long)a.layer * ws.pool_slots * ws.n_kv_heads + x.g) * D + ch * 8;
      const uint16_t *kb = static_cast<const uint16_t *>(ws.k_pool) + head0;
      const uint16_t *vb = static_cast<const uint16_t *>(ws.v_pool) + head0;
      const int ntiles = x.k1 > x.k0 ? (x.k1 - x.k0 + kXT - 1) / kXT : 0;
      // gathers: rows lane, lane + 32; TMA: lanes j, j + 4 hold piece j's page id
      int raw[2] = {raw_at(x.k0 + (TMA ? 16 * (lane & 3) : lane)),
                    TMA ? -1 : raw_at(x.k0 + lane + 32)};
      for (int tile = 0; tile < ntiles; ++tile, ++k) {
        const int s = k % kXStages, r = k / kXStages;
        if ((r > 0 && !mbar_wait_bounded(&empty[s], (r - 1) & 1)) || s_abort) {
          aborted = true;
          break;
        }
        const int t0 = x.k0 + tile * kXT;
        if constexpr (TMA) {
          // one box per 16-token piece and pool; a bad page loads the
          // in-range slot 0 and flags the stage
          const int np = min(4, (x.k1 - t0 + 15) / 16);
          const int j = lane & 3;
          int kind = 0, slot0 = 0;
          if (lane < 8 && j < np) {
            const long long s0 = slot_from_raw(ws, pl, raw[0], t0 + 16 * j, kind);
            if (!kind) slot0 = (int)s0;
          }
          const int nx = raw_at(t0 + kXT + 16 * j);
          const int bad = __reduce_or_sync(0xffffffffu, kind);
          if (lane == 0) {
            flags[s] = bad;
            if (bad) atomicOr(ws.err, bad);
          }
          __syncwarp();
          if (lane < 8 && j < np)
            xtma4(ring + s * C::STAGE + j * 2 * C::PIECE + (lane >> 2) * C::PIECE,
                  lane < 4 ? &tmk : &tmv, a.layer * ws.pool_slots + slot0, x.g, &full[s]);
          if (lane == 0) mbar_arrive_expect_tx(&full[s], np * (uint32_t)(2 * C::PIECE));
          raw[0] = nx;
          continue;
        }
        int kind = 0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int t = t0 + lane + 32 * h;
          // a bad table row reads as raw -1: a page error
          const int sl = t < x.k1 ? (int)slot_from_raw(ws, pl, raw[h], t, kind) : -1;
          s_slot[s][lane + 32 * h] = sl;
        }
        // the next tile's index entries load while this tile's copies issue
        const int nx[2] = {raw_at(t0 + kXT + lane), raw_at(t0 + kXT + lane + 32)};
        const int bad = __reduce_or_sync(0xffffffffu, kind);
        if (lane == 0) {
          flags[s] = bad;
          if (bad) atomicOr(ws.err, bad);
        }
        __syncwarp();
        const uint32_t kt = ring + s * C::STAGE, vt = kt + C::PIECE;
#pragma unroll 8
        for (int i = 0; i < kXT / RPI; ++i) {
          const int row = i * RPI + sub;
          const int sl = s_slot[s][row];
          const long long e = sl >= 0 ? sl * slot_elems : 0;
          const uint32_t off = xoff<D>(row, ch);
          xcp16(kt + off, kb + e, sl >= 0 ? 16 : 0);
          xcp16(vt + off, vb + e, sl >= 0 ? 16 : 0);
        }
        asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(
                         smem_addr(&full[s]))
                     : "memory");
        if (lane == 0) mbar_arrive(&full[s]);
        raw[0] = nx[0];
        raw[1] = nx[1];
      }
    }
    if (aborted) {
      if (lane == 0) {
        s_abort = 1;
        atomicOr(ws.err, PKV_DEVERR_TIMEOUT);
      }
      for (int kk = max(0, k - kXStages); kk < k; ++kk)
        mbar_wait_bounded(&full[kk % kXStages], (kk / kXStages) & 1);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    return;
  }

  // ---------------------------------------------------------- consumers ----
  const int grp = lane >> 2, tig = lane & 3;
  const float qk_scale = a.scale * kLog2e;
  const int mi = lane >> 3, rr = lane & 7;
  int k = 0;
  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    const XUnit x = xunit(a, u, TQ, jmax);
    if (!x.live) continue;
    // this lane's two rows (grp, grp + 8 of the warp's 16)
    int pos[2], qrow[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int row = 16 * warp + grp + 8 * e;
      const int i = x.j * TQ + row / G;
      const bool valid = i < x.n;
      pos[e] = !valid ? -1 : (a.flags & PKV_FLAG_EXTEND_FULL) ? x.L - 1 : x.L - x.n + i;
      qrow[e] = valid ? (x.q0 + i) * Hq + x.g * G + row % G : -1;
    }
    // the warp's last attended key (tiles past it are skipped) and the first
    // valid row's position (tiles wholly before it need no mask; rows past
    // the block's tokens, pos -1, are never written)
    int wpos = max(pos[0], pos[1]);
    wpos = __reduce_max_sync(0xffffffffu, wpos);
    int wmin = min(pos[0] < 0 ? INT_MAX : pos[0], pos[1] < 0 ? INT_MAX : pos[1]);
    wmin = __reduce_min_sync(0xffffffffu, wmin);
    // Q as the A operand: qa[ks] = {Q[r0][c..], Q[r1][c..], Q[r0][c+8..], Q[r1][c+8..]},
    // c = 16 ks + 2 tig
    uint32_t qa[C::KSTEPS][4];
    {
      const uint32_t *q32 = static_cast<const uint32_t *>(a.q);
#pragma unroll
      for (int ks = 0; ks < C::KSTEPS; ++ks) {
        const int c2 = (16 * ks + 2 * tig) / 2;
        qa[ks][0] = qrow[0] >= 0 ? q32[(long long)qrow[0] * (D / 2) + c2] : 0u;
        qa[ks][1] = qrow[1] >= 0 ? q32[(long long)qrow[1] * (D / 2) + c2] : 0u;
        qa[ks][2] = qrow[0] >= 0 ? q32[(long long)qrow[0] * (D / 2) + c2 + 4] : 0u;
        qa[ks][3] = qrow[1] >= 0 ? q32[(long long)qrow[1] * (D / 2) + c2 + 4] : 0u;
      }
    }
    float oacc[C::ND][4];
#pragma unroll
    for (int nd = 0; nd < C::ND; ++nd) oacc[nd][0] = oacc[nd][1] = oacc[nd][2] = oacc[nd][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    int bad = 0;
    const int ntiles = x.k1 > x.k0 ? (x.k1 - x.k0 + kXT - 1) / kXT : 0;
    for (int tile = 0; tile < ntiles; ++tile, ++k) {
      const int s = k % kXStages;
      bool ok = false;
      if (!s_abort) {
        ok = mbar_wait_bounded(&full[s], (k / kXStages) & 1);
        if (!ok && lane == 0) {
          s_abort = 1;
          atomicOr(ws.err, PKV_DEVERR_TIMEOUT);
        }
      }
      const int t0 = x.k0 + tile * kXT;
      if (TMA && t0 + kXT > x.k1) {
        // The boxes bring whole pieces: V rows past the unit's last key hold
        // whatever the pool (or an earlier tile) held, and P = 0 there does
        // not cancel a NaN.  Clear them (every consumer warp reaches this
        // for the same tile), then order the writes before the next boxes.
        const int first = x.k1 - t0;
        const uint32_t vt0 = ring + s * C::STAGE + C::PIECE;
        for (int i = tid; i < (kXT - first) * (D / 8); i += kXW * 32) {
          const int r = first + i / (D / 8), c = i % (D / 8);
          asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(vt0 + xoff<D>(r, c)),
                       "r"(0u)
                       : "memory");
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        named_sync(1, kXW * 32);
      }
      if (!ok) {
        bad = 1;
      } else if ((bad |= flags[s]) == 0 && t0 <= wpos) {
        const uint32_t kt = ring + s * C::STAGE, vt = kt + C::PIECE;
        // ---- S = Q K^T: 8 n-tiles of 8 keys ----
        float sc[8][4];
#pragma unroll
        for (int n = 0; n < 8; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < C::KSTEPS; ks += 2) {
#pragma unroll
          for (int n = 0; n < 8; ++n) {
            // matrices: keys 8n..8n+7 x dims of chunks 2ks + mi (k-steps ks, ks + 1)
            uint32_t b0, b1, b2, b3;
            ldsm_x4(kt + xoff<D>(8 * n + rr, 2 * ks + mi), b0, b1, b2, b3);
            mma_bf16_16816(sc[n], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
            mma_bf16_16816(sc[n], qa[ks + 1][0], qa[ks + 1][1], qa[ks + 1][2], qa[ks + 1][3], b2,
                           b3);
          }
        }
        // ---- causal mask, online softmax per row (log2 units) ----
        float mx[2] = {-INFINITY, -INFINITY};
        if (t0 + kXT - 1 <= wmin) {  // every key of the tile is attended by every row
#pragma unroll
          for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              sc[n][c] *= qk_scale;
              mx[c >> 1] = fmaxf(mx[c >> 1], sc[n][c]);
            }
        } else {
#pragma unroll
          for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int e = c >> 1;
              const int key = t0 + 8 * n + 2 * tig + (c & 1);
              const float v = key <= pos[e] ? sc[n][c] * qk_scale : -INFINITY;
              sc[n][c] = v;
              mx[e] = fmaxf(mx[e], v);
            }
        }
        float al[2], mref[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 1));
          mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 2));
          const float mn = fmaxf(m_run[e], mx[e]);
          mref[e] = mn == -INFINITY ? 0.f : mn;  // a row with nothing attended yet
          al[e] = exp2f(m_run[e] - mref[e]);
          m_run[e] = mn;
          l_run[e] *= al[e];
        }
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float p = exp2f(sc[n][c] - mref[c >> 1]);
            sc[n][c] = p;
            l_run[c >> 1] += p;
          }
#pragma unroll
        for (int nd = 0; nd < C::ND; ++nd) {
          oacc[nd][0] *= al[0];
          oacc[nd][1] *= al[0];
          oacc[nd][2] *= al[1];
          oacc[nd][3] *= al[1];
        }
        // ---- O += P V: 4 k-steps of 16 keys, P rounded to bf16 ----
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          uint32_t ph[4];
#pragma unroll
          for (int f = 0; f < 4; ++f) {
            // f: (row grp, keys lo), (row grp+8, keys lo), (row grp, keys hi), (row grp+8, keys hi)
            const float *src = sc[2 * kk + (f >> 1)] + 2 * (f & 1);
            ph[f] = pack_bf16x2(src[0], src[1]);
          }
#pragma unroll
          for (int nd = 0; nd < C::ND; nd += 2) {
            // matrices: keys 16kk + 8 (mi & 1) .. + 7 x dims of chunk nd + (mi >> 1)
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(vt + xoff<D>(16 * kk + 8 * (mi & 1) + rr, nd + (mi >> 1)), b0, b1, b2, b3);
            mma_bf16_16816(oacc[nd], ph[0], ph[1], ph[2], ph[3], b0, b1);
            mma_bf16_16816(oacc[nd + 1], ph[0], ph[1], ph[2], ph[3], b2, b3);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    // ---- normalise and write this lane's rows ----
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float l = l_run[e];
      l += __shfl_xor_sync(0xffffffffu, l, 1);
      l += __shfl_xor_sync(0xffffffffu, l, 2);
      if (qrow[e] < 0) continue;
      // a failed unit is written as zeros whatever its tiles held
      const bool zero = bad || !(l > 0.f);
      const float inv = zero ? 0.f : 1.f / l;
      if (a.S > 1) {
        // split partial: normalised o and (m, l) in natural-log units; a
        // failed split is marked l = -1 so the merge writes the row as zeros
        const long long pr = (long long)qrow[e] * a.S + x.c;
        float *op = ws.o_part + pr * D + 2 * tig;
#pragma unroll
        for (int nd = 0; nd < C::ND; ++nd)
          *reinterpret_cast<float2 *>(op + 8 * nd) =
              make_float2(zero ? 0.f : oacc[nd][2 * e] * inv, zero ? 0.f : oacc[nd][2 * e + 1] * inv);
        if (tig == 0) {
          ws.ml_part[pr * 2] = zero ? -INFINITY : m_run[e] * kLn2;
          ws.ml_part[pr * 2 + 1] = bad ? -1.f : (zero ? 0.f : l);
        }
        continue;
      }
      if ((a.flags & PKV_FLAG_WRITE_LSE) && tig == 0)
        ws.lse[qrow[e]] = zero ? -INFINITY : m_run[e] * kLn2 + logf(l);
      const long long o = (long long)qrow[e] * D + 2 * tig;
#pragma unroll
      for (int nd = 0; nd < C::ND; ++nd) {
        const float v0 = zero ? 0.f : oacc[nd][2 * e] * inv;
        const float v1 = zero ? 0.f : oacc[nd][2 * e + 1] * inv;
        if (a.flags & PKV_FLAG_OUT_F32) {
          *reinterpret_cast<float2 *>(static_cast<float *>(a.out) + o + 8 * nd) =
              make_float2(v0, v1);
        } else {
          *reinterpret_cast<uint32_t *>(static_cast<uint16_t *>(a.out) + o + 8 * nd) =
              pack_bf16x2(v0, v1);
        }
      }
    }
  }
}

// Merge of the split partials: one warp per (new token, query head) of
// request b = blockIdx.y: M = max over non-empty splits of m_s, w_s = l_s
// exp(m_s - M), out = sum w_s o_s / sum w_s; zeros when no split has a key
// or one failed (l = -1).  The splits' (m, l) are read one per lane and the
// partial rows with independent loads (merge_row), so a row costs a few
// memory round trips, not two per split.
template <int D>
__global__ void __launch_bounds__(128)
    extend_merge_kernel(const __grid_constant__ pkv_workspace ws, const int *qo_indptr,
                        int max_qo_len, int S, void *out, int flags) {
  pdl_wait();
  pdl_trigger();
  constexpr int NV = D / 4;  // float4 vectors per row
  const int b = blockIdx.y;
  const int q0 = qo_indptr[b], n = qo_indptr[b + 1] - q0, L = ws.seq_lens[b];
  const long long cap = len_cap(ws);
  const bool fits = (flags & PKV_FLAG_EXTEND_FULL) || n <= L;  // as the attention kernel
  bool ok = n >= 0 && fits && n <= max_qo_len && q0 >= 0 && q0 + n <= qo_indptr[gridDim.y] &&
            (long long)L <= cap && (long long)q0 + n <= (long long)gridDim.y * max_qo_len;
  if (ok && ws.index_mode == PKV_IDX_FLAT) {
    const int base = ws.kv_indptr[b];
    ok = base >= 0 && (long long)base + L <= ws.max_total_tokens;
  }
  if (!ok) return;  // raised by the attention kernel
  const int Hq = ws.n_q_heads, lane = threadIdx.x & 31;
  for (int p = blockIdx.x * 4 + (threadIdx.x >> 5); p < n * Hq; p += gridDim.x * 4) {
    const long long row = (long long)(q0 + p / Hq) * Hq + p % Hq;
    const float *ml = ws.ml_part + row * S * 2;
    bool failed = false;
    for (int c = lane; c < S; c += 32) failed |= __ldcg(ml + 2 * c + 1) < 0.f;
    float M, den;
    float4 acc;
    merge_row<D>(ml, ws.o_part + row * S * D, S, lane, M, den, acc);
    const bool zero = __any_sync(0xffffffffu, failed) || !(den > 0.f);
    const float inv = zero ? 0.f : 1.f / den;
    if ((flags & PKV_FLAG_WRITE_LSE) && lane == 0) ws.lse[row] = zero ? -INFINITY : M + logf(den);
    if (lane < NV) {
      const float4 r = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
      if (flags & PKV_FLAG_OUT_F32) {
        reinterpret_cast<float4 *>(static_cast<float *>(out) + row * D)[lane] = r;
      } else {
        uint2 pk;
        pk.x = pack_bf16x2(r.x, r.y);
        pk.y = pack_bf16x2(r.z, r.w);
        reinterpret_cast<uint2 *>(static_cast<uint16_t *>(out) + row * D)[lane] = pk;
      }
    }
  }
}

// Two-way log-sum-exp merge (a cascade's shared-prefix and own-suffix
// results): one warp per row, two columns per lane and step.
__global__ void __launch_bounds__(128)
    merge_lse_kernel(int n_rows, int D, const float *o_a, const float *lse_a, const float *o_b,
                     const float *lse_b, void *out, float *lse_out, int flags) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  for (long long r = blockIdx.x * 4ll + (threadIdx.x >> 5); r < n_rows; r += gridDim.x * 4ll) {
    const float la = lse_a[r], lb = lse_b[r];
    const float M = fmaxf(la, lb);
    const bool none = M == -INFINITY;
    const float wa = (none || la == -INFINITY) ? 0.f : expf(la - M);
    const float wb = (none || lb == -INFINITY) ? 0.f : expf(lb - M);
    const float inv = none ? 0.f : 1.f / (wa + wb);
    for (int d = 2 * lane; d < D; d += 64) {
      const float2 x = *reinterpret_cast<const float2 *>(o_a + r * D + d);
      const float2 y = *reinterpret_cast<const float2 *>(o_b + r * D + d);
      const float v0 = none ? 0.f : (wa * x.x + wb * y.x) * inv;
      const float v1 = none ? 0.f : (wa * x.y + wb * y.y) * inv;
      if (flags & PKV_FLAG_OUT_F32)
        *reinterpret_cast<float2 *>(static_cast<float *>(out) + r * D + d) = make_float2(v0, v1);
      else
        *reinterpret_cast<uint32_t *>(static_cast<uint16_t *>(out) + r * D + d) =
            pack_bf16x2(v0, v1);
    }
    if (lse_out && lane == 0) lse_out[r] = none ? -INFINITY : M + logf(wa + wb);
  }
}

// Append: block (x, b) copies new tokens x, x + gridDim.x, ... of request b
// (K and V, every KV head) to the slots of their positions.
__global__ void __launch_bounds__(128)
    extend_append_kernel(const __grid_constant__ pkv_workspace ws, int layer,
                         const int *qo_indptr, int max_qo_len, const uint4 *k_new,
                         const uint4 *v_new) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.y;
  const int q0 = qo_indptr[b], n = qo_indptr[b + 1] - q0, L = ws.seq_lens[b];
  const long long cap = len_cap(ws);
  bool ok = n >= 0 && n <= L && n <= max_qo_len && q0 >= 0 && q0 + n <= qo_indptr[gridDim.y] &&
            (long long)L <= cap;
  long long base = 0;
  if (ok && ws.index_mode == PKV_IDX_FLAT) {
    base = ws.kv_indptr[b];
    ok = base >= 0 && base + L <= ws.max_total_tokens;
  } else if (ok) {
    const int row = ws.req_pool_indices[b];
    ok = row >= 0 && row < ws.max_reqs;
    base = ok ? (long long)row * ws.max_pages_per_req : 0;
  }
  if (!ok) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(ws.err, PKV_DEVERR_LEN);
    return;
  }
  const int P = ws.page_size;
  const int V16 = ws.n_kv_heads * ws.head_dim / 8;  // 16-byte vectors per token row
  for (int i = blockIdx.x; i < n; i += gridDim.x) {
    const int t = L - n + i;
    long long slot;
    if (ws.index_mode == PKV_IDX_FLAT) {
      const int s = ws.kv_indices[base + t];
      if (s < 0 || s >= ws.pool_slots) {
        if (threadIdx.x == 0) atomicOr(ws.err, PKV_DEVERR_SLOT);
        continue;
      }
      slot = s;
    } else {
      const int page = ws.page_table[base + t / P];
      if (page < 0 || page >= ws.pool_slots / P) {
        if (threadIdx.x == 0) atomicOr(ws.err, PKV_DEVERR_PAGE);
        continue;
      }
      slot = (long long)page * P + t % P;
    }
    const long long src = (long long)(q0 + i) * V16;
    const long long dst = ((long long)layer * ws.pool_slots + slot) * V16;
    uint4 *kp = static_cast<uint4 *>(ws.k_pool);
    uint4 *vp = static_cast<uint4 *>(ws.v_pool);
    for (int v = threadIdx.x; v < V16; v += blockDim.x) {
      kp[dst + v] = k_new[src + v];
      vp[dst + v] = v_new[src + v];
    }
  }
}

template <int D, int G>
cudaError_t launch_extend_one(const XArgs &a, cudaStream_t st) {
  using C = XCfg<D>;
  static int occ_cache[64] = {0};
  static int sms_cache[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int di = dev & 63;
  if (occ_cache[di] == 0) {
    auto kt = extend_mma_kernel<D, G, true>;
    auto kg = extend_mma_kernel<D, G, false>;
    e = cudaFuncSetAttribute(kt, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kg, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    int occ = 0, occ_g = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kt, kXThreads, C::SMEM);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_g, kg, kXThreads, C::SMEM);
    if (e != cudaSuccess) return e;
    occ = occ < occ_g ? occ : occ_g;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    sms_cache[di] = sms;
    occ_cache[di] = occ > 0 ? occ : 1;
  }
  constexpr int TQ = kXRows / G;
  const long long units =
      (long long)((a.max_qo_len + TQ - 1) / TQ) * a.S * a.batch * a.ws.n_kv_heads;
  if (units <= 0) return cudaSuccess;
  if (units > 0x7fffffffll) return cudaErrorInvalidValue;
  const long long cap = (long long)sms_cache[di] * occ_cache[di];
  const int grid = (int)(units < cap ? units : cap);
  const pkv_workspace &ws = a.ws;
  CUtensorMap tmk, tmv;
  memset(&tmk, 0, sizeof(tmk));
  memset(&tmv, 0, sizeof(tmv));
  const bool tma = ws.index_mode == PKV_IDX_PAGE_TABLE && ws.page_size % 16 == 0 &&
                   (long long)ws.n_layers * ws.pool_slots < 0x7fffffffll &&
                   xencode_pool_map(&tmk, ws.k_pool, ws, D / 64) &&
                   xencode_pool_map(&tmv, ws.v_pool, ws, D / 64);
  // Programmatic dependent launch when the grid leaves block slots free (its
  // start then overlaps the previous kernel's end: the cascade's prefix
  // attention, 36.4 -> 31.6 us per layer); a grid that fills every slot
  // launches plainly (early, its blocks only park: 3 % slower measured).
  if (grid < cap) {
    e = tma ? launch_pdl(extend_mma_kernel<D, G, true>, dim3(grid), dim3(kXThreads), C::SMEM,
                         st, a, tmk, tmv)
            : launch_pdl(extend_mma_kernel<D, G, false>, dim3(grid), dim3(kXThreads), C::SMEM,
                         st, a, tmk, tmv);
  } else {
    if (tma) extend_mma_kernel<D, G, true><<<grid, kXThreads, C::SMEM, st>>>(a, tmk, tmv);
    else extend_mma_kernel<D, G, false><<<grid, kXThreads, C::SMEM, st>>>(a, tmk, tmv);
    e = cudaGetLastError();
  }
  if (a.S > 1 && e == cudaSuccess) e = launch_extend_merge(a, D, st);
  return e;
}

}  // namespace

cudaError_t launch_extend_merge(const XArgs &a, int D, cudaStream_t st) {
  const pkv_workspace &ws = a.ws;
  const long long pairs = (long long)a.max_qo_len * ws.n_q_heads;
  const long long mblocks = (pairs + 3) / 4;
  const dim3 mgrid((unsigned)(mblocks < 1024 ? mblocks : 1024), (unsigned)a.batch);
  if (D == 128)
    return launch_pdl(extend_merge_kernel<128>, mgrid, dim3(128), 0, st, ws, a.qo_indptr,
                      a.max_qo_len, a.S, a.out, a.flags);
  if (D == 64)
    return launch_pdl(extend_merge_kernel<64>, mgrid, dim3(128), 0, st, ws, a.qo_indptr,
                      a.max_qo_len, a.S, a.out, a.flags);
  return cudaErrorNotSupported;
}

bool extend_supported(int head_dim, int group) {
  return (head_dim == 64 || head_dim == 128) &&
         (group == 1 || group == 2 || group == 4 || group == 8 || group == 16);
}

cudaError_t launch_extend(const pkv_workspace &ws, int batch, int layer, const int *qo_indptr,
                          int max_qo_len, const void *q, void *out, float scale, int num_splits,
                          int flags, cudaStream_t st) {
  XArgs a{ws, batch, layer, max_qo_len, flags & ~PKV_FLAG_EXTEND_WARP_MMA, num_splits, qo_indptr,
          q, out, scale};
  // the tcgen05 kernel where tensor-map boxes carry the pages; this file's
  // warp-level kernel for the rest (and by request)
  if (!(flags & PKV_FLAG_EXTEND_WARP_MMA) && extend_umma_supported(ws)) {
    const cudaError_t e = launch_extend_umma(a, st);
    if (e != cudaErrorNotSupported) return e;
  }
  const int D = ws.head_dim, G = ws.n_q_heads / ws.n_kv_heads;
#define PKV_X_CASE(DD, GG) \
  if (D == DD && G == GG) return launch_extend_one<DD, GG>(a, st);
  PKV_X_CASE(128, 1) PKV_X_CASE(128, 2) PKV_X_CASE(128, 4) PKV_X_CASE(128, 8)
  PKV_X_CASE(128, 16) PKV_X_CASE(64, 1) PKV_X_CASE(64, 2) PKV_X_CASE(64, 4)
  PKV_X_CASE(64, 8) PKV_X_CASE(64, 16)
#undef PKV_X_CASE
  return cudaErrorNotSupported;
}

cudaError_t launch_merge_lse(int n_rows, int head_dim, const float *o_a, const float *lse_a,
                             const float *o_b, const float *lse_b, void *out, float *lse_out,
                             int flags, cudaStream_t st) {
  const long long blocks = ((long long)n_rows + 3) / 4;
  return launch_pdl(merge_lse_kernel, dim3((unsigned)(blocks < 4096 ? blocks : 4096)), dim3(128),
                    0, st, n_rows, head_dim, o_a, lse_a, o_b, lse_b, out, lse_out, flags);
}

cudaError_t launch_extend_append(const pkv_workspace &ws, int batch, int layer,
                                 const int *qo_indptr, int max_qo_len, const void *k_new,
                                 const void *v_new, cudaStream_t st) {
  if (batch <= 0 || max_qo_len <= 0) return cudaSuccess;
  const dim3 grid((unsigned)min(max_qo_len, 64), (unsigned)batch);
  return launch_pdl(extend_append_kernel, grid, dim3(128), 0, st, ws, layer, qo_indptr,
                    max_qo_len, static_cast<const uint4 *>(k_new),
                    static_cast<const uint4 *>(v_new));
}

}  // namespace pkv
