// CUDA-core split-KV GQA decode attention (workspace.py page, bullets 1 and
// 14-16: the decode kernel and its split partial buffers).
//
// Work unit: (request b, KV head g, split c) over tokens [c*chunk,
// min((c+1)*chunk, L_b)), with chunk derived on the device from the live
// seq_lens (see split_chunk).  A persistent grid walks the units; each CTA's
// units form one stream of 32-token tiles.
//
// Data movement: warp 0 issues one bulk copy (TMA engine, cp.async.bulk) per
// K row and per V row of a tile, completing on a per-stage mbarrier; a
// 4-stage ring keeps ~64 KB per CTA in flight.  Page ids are read from the
// table by the issuing lanes and checked against the pool.
//
// Math: the KV head is read once per tile and reused for its whole group of
// G query heads.  Lanes are split into groups of D/8 lanes, one K/V row per
// group; each lane holds an 8-element slice of q (pre-scaled by
// scale*log2 e) for all G heads.  Scores are reduced across the group with a
// halving butterfly (G values in log2(G) + log2(D/8) shuffle rounds).  The
// softmax is online per tile in fp32 with exp2; the running output is kept
// per lane group and summed across groups at the end of the unit.
#include "kernels.cuh"

namespace pkv {

namespace {

constexpr int kThreads = 128;
constexpr int kWarps = 4;
constexpr int kT = 32;       // tokens per tile (one lane per token in the softmax)
constexpr int kStages = 4;   // tiles in flight per CTA

template <int D, int G>
struct Cfg {
  static constexpr int LPR = D / 8;             // lanes per row
  static constexpr int RPW = 32 / LPR;          // rows per warp per pass
  static constexpr int ROWS_PER_PASS = kWarps * RPW;
  static constexpr int PASSES = kT / ROWS_PER_PASS;
  static constexpr int ROW_BYTES = D * 2;
  static constexpr int TILE_BYTES = kT * ROW_BYTES;  // K or V of one tile
  static constexpr int HPW = (G + kWarps - 1) / kWarps;  // softmax heads per warp
  // dynamic shared memory layout (bytes)
  static constexpr int OFF_BAR = 0;                                  // kStages u64
  static constexpr int OFF_FLAG = 64;                                // kStages int
  static constexpr int OFF_KV = 128;                                 // stages
  static constexpr int OFF_SC = OFF_KV + kStages * 2 * TILE_BYTES;   // [kT][G] f32
  static constexpr int OFF_RED = OFF_SC + kT * G * 4;                // [kWarps][G][D] f32
  static constexpr int OFF_ALPHA = OFF_RED + kWarps * G * D * 4;     // [G] f32
  static constexpr int OFF_ML = OFF_ALPHA + 32;                      // [G][2] f32
  static constexpr int SMEM = OFF_ML + 2 * G * 4 + 64;
  static_assert(PASSES * ROWS_PER_PASS == kT, "tile must be a whole number of passes");
  static_assert(G <= LPR, "group reduce needs G <= D/8");
};

// Reduce G partial dot products across the LPR lanes of a row group.  Each
// halving round sends half of the remaining values to the partner lane, so
// every lane ends with the full sum for one head; `head` says which.
template <int LPR, int G>
__device__ __forceinline__ float group_reduce(float (&v)[G], int lane, int &head) {
  head = 0;
  int n = G;
#pragma unroll
  for (int d = LPR / 2; d >= 1; d >>= 1) {
    if (n > 1) {
      const int half = n / 2;
      const bool up = (lane & d) != 0;
#pragma unroll
      for (int i = 0; i < G / 2; ++i) {
        if (i < half) {
          const float keep = up ? v[half + i] : v[i];
          const float send = up ? v[i] : v[half + i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, d);
        }
      }
      if (up) head += half;
      n = half;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], d);
    }
  }
  return v[0];
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, d));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) x += __shfl_xor_sync(0xffffffffu, x, d);
  return x;
}

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
  const long long cap = len_cap(ws);
  if (L < 0 || (long long)L > cap) L = 0;  // flagged once per request by the c == 0 unit
  if (ws.index_mode == PKV_IDX_FLAT && L > 0) {
    const int base = ws.kv_indptr[x.b];
    if (base < 0 || (long long)base + L > ws.max_total_tokens) L = 0;
  }
  x.t0 = x.c * pl.chunk;
  x.t1 = min(x.t0 + pl.chunk, L);
  return x;
}

// Producer cursor over the CTA's tile stream (kept uniform across warp 0).
struct Cursor {
  Unit un;
  int i;       // next tile of un
  int ntiles;  // tiles of un
  bool done;
};

__device__ __forceinline__ void cursor_seek(const pkv_workspace &ws, const Plan &pl, Cursor &cu,
                                            int u) {
  for (; u < pl.n_units; u += gridDim.x) {
    cu.un = unit_at(ws, pl, u);
    if (cu.un.t0 < cu.un.t1) {
      cu.i = 0;
      cu.ntiles = (cu.un.t1 - cu.un.t0 + kT - 1) / kT;
      cu.done = false;
      return;
    }
  }
  cu.done = true;
}

template <int D, int G>
__device__ __forceinline__ void issue_tile(const DecodeArgs &a, const Plan &pl, Cursor &cu,
                                           int stage, uint8_t *smem, int lane) {
  using C = Cfg<D, G>;
  const pkv_workspace &ws = a.ws;
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR) + stage;
  int *flag = reinterpret_cast<int *>(smem + C::OFF_FLAG) + stage;
  uint8_t *kdst = smem + C::OFF_KV + (2 * stage) * C::TILE_BYTES;
  uint8_t *vdst = kdst + C::TILE_BYTES;

  const Unit &un = cu.un;
  const int tile0 = un.t0 + cu.i * kT;
  const int nvalid = min(kT, un.t1 - tile0);
  const int tok = tile0 + lane;
  const bool want = lane < nvalid;
  long long slot = -1;
  int kind = 0;
  if (want) {
    if (ws.index_mode == PKV_IDX_FLAT) {
      const int s = ws.kv_indices[ws.kv_indptr[un.b] + tok];
      if (s >= 0 && s < ws.pool_slots) slot = s;
      else kind = PKV_DEVERR_SLOT;
    } else {
      const int row = ws.req_pool_indices[un.b];
      if (row >= 0 && row < ws.max_reqs) {
        const int P = ws.page_size;
        const int page = ws.page_table[(long long)row * ws.max_pages_per_req + tok / P];
        if (page >= 0 && page < ws.pool_slots / P) slot = (long long)page * P + tok % P;
        else kind = PKV_DEVERR_PAGE;
      } else {
        kind = PKV_DEVERR_PAGE;
      }
    }
  }
  const unsigned ok = __ballot_sync(0xffffffffu, slot >= 0);
  const int bad_kind = __reduce_or_sync(0xffffffffu, kind);
  if (lane == 0) {
    *flag = bad_kind;
    if (bad_kind) atomicOr(ws.err, bad_kind);
    mbar_arrive_expect_tx(bar, __popc(ok) * 2u * C::ROW_BYTES);
  }
  __syncwarp();
  if (slot >= 0) {
    const long long row_elems =
        (((long long)a.layer * ws.pool_slots + slot) * ws.n_kv_heads + un.g) * D;
    const uint16_t *kp = static_cast<const uint16_t *>(ws.k_pool) + row_elems;
    const uint16_t *vp = static_cast<const uint16_t *>(ws.v_pool) + row_elems;
    bulk_g2s(kdst + lane * C::ROW_BYTES, kp, C::ROW_BYTES, bar);
    bulk_g2s(vdst + lane * C::ROW_BYTES, vp, C::ROW_BYTES, bar);
  }
  // advance
  if (++cu.i == cu.ntiles) cursor_seek(ws, pl, cu, cu.un.u + gridDim.x);
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads) decode_simt_kernel(const DecodeArgs a) {
  using C = Cfg<D, G>;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_max_len;
  const pkv_workspace &ws = a.ws;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Hq = ws.n_q_heads;

  // Prologue: split length from the batch's longest (valid) request.
  if (tid == 0) s_max_len = 0;
  __syncthreads();
  {
    int mx = 0;
    const long long cap = len_cap(ws);
    for (int b = tid; b < a.batch; b += kThreads) {
      const int L = ws.seq_lens[b];
      if (L >= 0 && (long long)L <= cap) mx = max(mx, L);
      else if (blockIdx.x == 0) atomicOr(ws.err, PKV_DEVERR_LEN);
      if (blockIdx.x == 0 && ws.index_mode == PKV_IDX_FLAT && L > 0) {
        const int base = ws.kv_indptr[b];
        if (base < 0 || (long long)base + L > ws.max_total_tokens)
          atomicOr(ws.err, PKV_DEVERR_TOTAL);
      }
    }
    mx = __reduce_max_sync(0xffffffffu, mx);
    if (lane == 0) atomicMax(&s_max_len, mx);
  }
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  __syncthreads();

  Plan pl;
  pl.batch = a.batch;
  pl.hkv = ws.n_kv_heads;
  pl.S = a.num_splits;
  pl.chunk = split_chunk(s_max_len, a.num_splits, ws.page_size);
  pl.n_units = pl.S * pl.batch * pl.hkv;
  const bool direct = pl.S == 1;

  // Producer: warp 0 fills the ring.
  Cursor pc;
  int issued = 0;
  if (warp == 0) {
    cursor_seek(ws, pl, pc, blockIdx.x);
    while (!pc.done && issued < kStages) {
      issue_tile<D, G>(a, pl, pc, issued % kStages, smem, lane);
      ++issued;
    }
  }

  const int *flags = reinterpret_cast<const int *>(smem + C::OFF_FLAG);
  float *sc = reinterpret_cast<float *>(smem + C::OFF_SC);
  float *red = reinterpret_cast<float *>(smem + C::OFF_RED);
  float *s_alpha = reinterpret_cast<float *>(smem + C::OFF_ALPHA);
  float *s_ml = reinterpret_cast<float *>(smem + C::OFF_ML);
  const int j = lane % C::LPR;               // d-slice of this lane: [8j, 8j+8)
  const int rsub = lane / C::LPR;            // row within the warp's pass
  const float qscale = a.scale * kLog2e;

  int k = 0;  // consumed stream items
  bool aborted = false;
  for (int u = blockIdx.x; u < pl.n_units; u += gridDim.x) {
    const Unit un = unit_at(ws, pl, u);
    const int hq0 = un.g * G;
    if (un.t0 >= un.t1) {
      // Empty split (past the request's end, or an empty request).
      if (direct) {
        for (int i = tid; i < G * D; i += kThreads) {
          const long long o = ((long long)un.b * Hq + hq0) * D + i;
          if (a.flags & PKV_FLAG_OUT_F32) static_cast<float *>(ws.out)[o] = 0.f;
          else static_cast<uint16_t *>(ws.out)[o] = 0;
        }
        if ((a.flags & PKV_FLAG_WRITE_LSE) && ws.lse && tid < G)
          ws.lse[(long long)un.b * Hq + hq0 + tid] = -INFINITY;
      } else if (tid < G) {
        const long long o = (((long long)un.b * Hq + hq0 + tid) * pl.S + un.c) * 2;
        ws.ml_part[o] = -INFINITY;
        ws.ml_part[o + 1] = 0.f;
      }
      continue;
    }
    const int ntiles = (un.t1 - un.t0 + kT - 1) / kT;

    // q slice for all G heads, pre-scaled into log2 units.
    float q[G][8];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const uint16_t *qp = static_cast<const uint16_t *>(a.q) +
                           ((long long)un.b * Hq + hq0 + h) * D + j * 8;
      float f[8];
      unpack8(*reinterpret_cast<const uint4 *>(qp), f);
#pragma unroll
      for (int e = 0; e < 8; ++e) q[h][e] = f[e] * qscale;
    }
    float acc[G][8];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[h][e] = 0.f;
    float m_run[C::HPW], l_run[C::HPW];
#pragma unroll
    for (int i = 0; i < C::HPW; ++i) {
      m_run[i] = -INFINITY;
      l_run[i] = 0.f;
    }
    int unit_bad = 0;

    for (int it = 0; it < ntiles; ++it, ++k) {
      const int stage = k % kStages;
      const uint32_t parity = (k / kStages) & 1;
      const bool ok = mbar_wait_bounded(&bars[stage], parity);
      if (__syncthreads_or(!ok)) {
        if (tid == 0) atomicOr(ws.err, PKV_DEVERR_TIMEOUT);
        aborted = true;
        break;
      }
      unit_bad |= flags[stage];
      const uint8_t *kt = smem + C::OFF_KV + (2 * stage) * C::TILE_BYTES;
      const uint8_t *vt = kt + C::TILE_BYTES;
      const int nvalid = min(kT, un.t1 - (un.t0 + it * kT));

      // ---- scores: s[t][h] = q_h . k_t (log2 units) ----
#pragma unroll
      for (int p = 0; p < C::PASSES; ++p) {
        const int row = p * C::ROWS_PER_PASS + warp * C::RPW + rsub;
        float part[G];
        if (row < nvalid) {
          float kf[8];
          unpack8(*reinterpret_cast<const uint4 *>(kt + row * C::ROW_BYTES + j * 16), kf);
#pragma unroll
          for (int h = 0; h < G; ++h) {
            float s = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) s = fmaf(q[h][e], kf[e], s);
            part[h] = s;
          }
        } else {
#pragma unroll
          for (int h = 0; h < G; ++h) part[h] = 0.f;
        }
        int head;
        const float s = group_reduce<C::LPR, G>(part, lane, head);
        if (row < nvalid && (j % (C::LPR / G)) == 0) sc[row * G + head] = s;
      }
      __syncthreads();

      // ---- online softmax over the tile: lane = token, warp owns heads ----
#pragma unroll
      for (int i = 0; i < C::HPW; ++i) {
        const int h = warp + i * kWarps;
        if (h < G) {
          const float s = lane < nvalid ? sc[lane * G + h] : -INFINITY;
          const float m_new = fmaxf(m_run[i], warp_max(s));
          const float pr = lane < nvalid ? exp2f(s - m_new) : 0.f;
          sc[lane * G + h] = pr;
          const float alpha = exp2f(m_run[i] - m_new);
          l_run[i] = l_run[i] * alpha + warp_sum(pr);
          m_run[i] = m_new;
          if (lane == 0) s_alpha[h] = alpha;
        }
      }
      __syncthreads();

      // ---- o += p . V ----
      float al[G];
#pragma unroll
      for (int h = 0; h < G; ++h) al[h] = s_alpha[h];
#pragma unroll
      for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[h][e] *= al[h];
#pragma unroll
      for (int p = 0; p < C::PASSES; ++p) {
        const int row = p * C::ROWS_PER_PASS + warp * C::RPW + rsub;
        if (row < nvalid) {
          float vf[8];
          unpack8(*reinterpret_cast<const uint4 *>(vt + row * C::ROW_BYTES + j * 16), vf);
          float pr[G];
#pragma unroll
          for (int h = 0; h < G; ++h) pr[h] = sc[row * G + h];
#pragma unroll
          for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[h][e] = fmaf(pr[h], vf[e], acc[h][e]);
        }
      }
      __syncthreads();  // stage and score buffers are free again

      if (warp == 0 && !pc.done) {
        issue_tile<D, G>(a, pl, pc, stage, smem, lane);
        ++issued;
      }
    }
    if (aborted) break;

    // ---- combine the row groups, normalise, write ----
#pragma unroll
    for (int off = C::LPR; off < 32; off <<= 1)
#pragma unroll
      for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], off);
    if (lane < C::LPR) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float4 *dst = reinterpret_cast<float4 *>(red + (warp * G + h) * D + j * 8);
        dst[0] = make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
        dst[1] = make_float4(acc[h][4], acc[h][5], acc[h][6], acc[h][7]);
      }
    }
#pragma unroll
    for (int i = 0; i < C::HPW; ++i) {
      const int h = warp + i * kWarps;
      if (h < G && lane == 0) {
        s_ml[2 * h] = m_run[i];
        s_ml[2 * h + 1] = l_run[i];
      }
    }
    const int bad = __syncthreads_or(unit_bad);
    for (int i = tid; i < G * D; i += kThreads) {
      const int h = i / D;
      float o = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) o += red[w * G * D + i];
      const float l = s_ml[2 * h + 1];
      o = bad ? 0.f : o / l;
      if (direct) {
        const long long off = ((long long)un.b * Hq + hq0) * D + i;
        if (a.flags & PKV_FLAG_OUT_F32) static_cast<float *>(ws.out)[off] = o;
        else static_cast<uint16_t *>(ws.out)[off] = (uint16_t)f32_to_bf16_bits(o);
      } else {
        const int d = i - h * D;
        ws.o_part[(((long long)un.b * Hq + hq0 + h) * pl.S + un.c) * D + d] = o;
      }
    }
    if (tid < G) {
      const float m = s_ml[2 * tid] * kLn2;  // back to natural-log units
      const float l = s_ml[2 * tid + 1];
      if (direct) {
        if ((a.flags & PKV_FLAG_WRITE_LSE) && ws.lse)
          ws.lse[(long long)un.b * Hq + hq0 + tid] = bad ? -INFINITY : m + logf(l);
      } else {
        const long long o = (((long long)un.b * Hq + hq0 + tid) * pl.S + un.c) * 2;
        ws.ml_part[o] = bad ? -INFINITY : m;
        ws.ml_part[o + 1] = bad ? 0.f : l;
      }
    }
    __syncthreads();  // red / s_ml reused by the next unit
  }

  // After a timeout, wait (bounded) for the copies still in flight so none
  // lands in shared memory after the CTA has exited.
  if (aborted) {
    for (int kk = k; kk < issued; ++kk) {
      mbar_wait_bounded(&bars[kk % kStages], (kk / kStages) & 1);
    }
  }
}

template <int D, int G>
cudaError_t launch_one(const DecodeArgs &a, cudaStream_t st) {
  using C = Cfg<D, G>;
  auto kern = decode_simt_kernel<D, G>;
  static int occ_cache[64] = {0};
  static int sms_cache[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int di = dev & 63;
  if (occ_cache[di] == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    int occ = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, C::SMEM);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    sms_cache[di] = sms;
    occ_cache[di] = occ > 0 ? occ : 1;
  }
  const long long units = (long long)a.num_splits * a.batch * a.ws.n_kv_heads;
  const long long cap = (long long)sms_cache[di] * occ_cache[di];
  const int grid = (int)(units < cap ? units : cap);
  if (grid <= 0) return cudaSuccess;
  kern<<<grid, kThreads, C::SMEM, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

bool decode_simt_supported(int head_dim, int group) {
  return (head_dim == 64 || head_dim == 128) &&
         (group == 1 || group == 2 || group == 4 || group == 8);
}

cudaError_t launch_decode_simt(const DecodeArgs &a, cudaStream_t st) {
  const int D = a.ws.head_dim, G = a.ws.n_q_heads / a.ws.n_kv_heads;
  if (D == 128) {
    switch (G) {
      case 1: return launch_one<128, 1>(a, st);
      case 2: return launch_one<128, 2>(a, st);
      case 4: return launch_one<128, 4>(a, st);
      case 8: return launch_one<128, 8>(a, st);
    }
  } else if (D == 64) {
    switch (G) {
      case 1: return launch_one<64, 1>(a, st);
      case 2: return launch_one<64, 2>(a, st);
      case 4: return launch_one<64, 4>(a, st);
      case 8: return launch_one<64, 8>(a, st);
    }
  }
  return cudaErrorNotSupported;
}

}  // namespace pkv
