// Definitions shared by the two paged extend (prefill) attention kernels:
// the warp-level one (extend_mma.cu) and the tcgen05 one (extend_umma.cu).
// Both take the same arguments, enumerate the same units and write the same
// outputs; the split merge and the tensor-map encoder live here too.
#pragma once

#include <cuda.h>

#include <utility>

#include "decode_plan.cuh"

namespace pkv {

constexpr int kXT = 64;  // keys per tile (split chunks are whole tiles)

struct XArgs {
  pkv_workspace ws;
  int batch, layer, max_qo_len, flags;
  int S;  // splits of each unit's key range (1: rows written to out directly)
  const int *qo_indptr;
  const void *q;
  void *out;
  float scale;
};

// One unit: request b's query block j for KV head g.
struct XUnit {
  int b, g, j, c;
  int n;       // new tokens of the request
  int L;       // its cached length (new tokens included)
  int q0;      // qo_indptr[b]
  int kend;    // the block's rows attend keys 0 .. kend - 1 at most
  int k0, k1;  // keys of split c: [k0, k1) (empty when k0 >= k1)
  bool live;   // valid request and a non-empty query block
};

// Unit u = (query block j, split c, request b, KV head g), j descending.
// Request b's new-token count and length are checked; PKV_DEVERR_LEN is
// raised once per request (by the unit with g, j and c all 0).  Split c of a
// block covers keys [c * chunk, (c + 1) * chunk) of its causal range,
// chunk = ceil(kend / S) rounded up to a whole tile.
__device__ __forceinline__ XUnit xunit(const XArgs &a, int u, int tq, int jmax) {
  const pkv_workspace &ws = a.ws;
  const int bh = a.batch * ws.n_kv_heads;
  XUnit x;
  const int jj = u / (bh * a.S), rs = u - jj * bh * a.S;
  x.c = rs / bh;
  const int r = rs - x.c * bh;
  x.b = r / ws.n_kv_heads;
  x.g = r - x.b * ws.n_kv_heads;
  x.j = jmax - 1 - jj;
  x.q0 = a.qo_indptr[x.b];
  x.n = a.qo_indptr[x.b + 1] - x.q0;
  x.L = ws.seq_lens[x.b];
  const long long cap = len_cap(ws);
  // full mode: the query rows are not tokens of the context, so n_b may exceed L_b
  const bool fits = (a.flags & PKV_FLAG_EXTEND_FULL) || x.n <= x.L;
  bool ok = x.n >= 0 && fits && x.n <= a.max_qo_len && x.q0 >= 0 &&
            x.q0 + x.n <= a.qo_indptr[a.batch] && (long long)x.L <= cap;
  if (ok && ws.index_mode == PKV_IDX_FLAT) {
    const int base = ws.kv_indptr[x.b];
    ok = base >= 0 && (long long)base + x.L <= ws.max_total_tokens;
  }
  // split partials and lse rows live in the workspace, sized for batch *
  // max_qo_len new tokens: a request whose rows lie past that (qo_indptr
  // running on past an invalid request) is rejected, not written
  if (ok && (a.S > 1 || (a.flags & PKV_FLAG_WRITE_LSE)))
    ok = (long long)x.q0 + x.n <= (long long)a.batch * a.max_qo_len;
  if (!ok && x.g == 0 && x.j == 0 && x.c == 0 && (threadIdx.x & 31) == 0)
    atomicOr(ws.err, PKV_DEVERR_LEN);
  x.live = ok && x.j * tq < x.n;
  x.kend = !x.live ? 0 : (a.flags & PKV_FLAG_EXTEND_FULL) ? x.L
                                                             : x.L - x.n + min(x.n, (x.j + 1) * tq);
  const int chunk = ((x.kend + a.S - 1) / a.S + kXT - 1) / kXT * kXT;
  x.k0 = x.c * chunk;
  x.k1 = min(x.kend, x.k0 + chunk);
  return x;
}

using XTmapEncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// 4-D view of a pool [NL * pool_slots, Hkv, D] as (64 columns, slot, 64-column
// half, KV head): a box of 64 x 16 x box_halves x 1 is one 16-token piece of
// one head (box_halves = D / 64: both halves, landing 128B-swizzled as
// [half][token][64 columns]; box_halves = 1: the half at the box's third
// coordinate, as [token][64 columns]).
inline bool xencode_pool_map(CUtensorMap *m, void *base, const pkv_workspace &ws,
                             int box_halves) {
  static XTmapEncodeFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<XTmapEncodeFn>(p);
  }
  if (!fn) return false;
  const cuuint64_t D = (cuuint64_t)ws.head_dim, H = (cuuint64_t)ws.n_kv_heads;
  const cuuint64_t dims[4] = {64, (cuuint64_t)ws.n_layers * (cuuint64_t)ws.pool_slots, D / 64, H};
  const cuuint64_t strides[3] = {H * D * 2, 128, D * 2};
  const cuuint32_t box[4] = {64, 16, (cuuint32_t)box_halves, 1};
  const cuuint32_t elem[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box, elem,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Whether tensor-map boxes can carry the workspace's pages (whole 16-token
// pieces inside one page, slot coordinates that fit an int).
inline bool xtma_pages(const pkv_workspace &ws) {
  return ws.index_mode == PKV_IDX_PAGE_TABLE && ws.page_size % 16 == 0 &&
         (long long)ws.n_layers * ws.pool_slots < 0x7fffffffll;
}

// Launch with programmatic dependent launch allowed (the kernels wait for
// the previous kernel on the stream at entry).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// The split merge after an extend launch with a.S > 1 (extend_mma.cu).
cudaError_t launch_extend_merge(const XArgs &a, int D, cudaStream_t st);

// The tcgen05 kernel (extend_umma.cu): whether it serves the shape, and its
// launch (cudaErrorNotSupported: the caller takes the warp-level kernel).
bool extend_umma_supported(const pkv_workspace &ws);
cudaError_t launch_extend_umma(const XArgs &a, cudaStream_t st);

}  // namespace pkv
