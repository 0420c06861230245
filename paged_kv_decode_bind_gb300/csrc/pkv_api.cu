// C-ABI entry points of libpkv (declared in include/pkv.h): host-side
// validation, then kernel launches on the caller's stream.  Nothing here
// allocates, synchronises or reads device memory.
#include <cstring>

#include "kernels.cuh"

using namespace pkv;

namespace pkv {
// extend_mma.cu
cudaError_t launch_extend(const pkv_workspace &ws, int batch, int layer, const int *qo_indptr,
                          int max_qo_len, const void *q, void *out, float scale, int num_splits,
                          int flags, cudaStream_t st);
cudaError_t launch_extend_append(const pkv_workspace &ws, int batch, int layer,
                                 const int *qo_indptr, int max_qo_len, const void *k_new,
                                 const void *v_new, cudaStream_t st);
bool extend_supported(int head_dim, int group);
bool extend_umma_supported(const pkv_workspace &ws);  // extend_umma.cu
cudaError_t launch_merge_lse(int n_rows, int head_dim, const float *o_a, const float *lse_a,
                             const float *o_b, const float *lse_b, void *out, float *lse_out,
                             int flags, cudaStream_t st);
}  // namespace pkv

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// ml_part is read as (m, l) float pairs
bool aligned8(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; }

// Shape checks shared by every entry point.
pkv_status check_shape(const pkv_workspace *ws) {
  if (!ws) return PKV_ERR_INVALID;
  if (ws->n_layers <= 0 || ws->pool_slots <= 0 || ws->n_q_heads <= 0 || ws->n_kv_heads <= 0 ||
      ws->head_dim <= 0 || ws->page_size <= 0 || ws->max_batch < 0 || ws->max_reqs <= 0 ||
      ws->max_pages_per_req <= 0 || ws->max_splits <= 0 || ws->max_seq_len < 0)
    return PKV_ERR_INVALID;
  if (ws->n_q_heads % ws->n_kv_heads != 0) return PKV_ERR_INVALID;
  if (ws->pool_slots % ws->page_size != 0) return PKV_ERR_INVALID;
  if (ws->index_mode != PKV_IDX_PAGE_TABLE && ws->index_mode != PKV_IDX_FLAT)
    return PKV_ERR_INVALID;
  if (ws->index_mode == PKV_IDX_FLAT && ws->page_size != 1) return PKV_ERR_INVALID;
  if (ws->head_dim % 8 != 0) return PKV_ERR_UNSUPPORTED;
  if (!ws->err) return PKV_ERR_INVALID;
  return PKV_OK;
}

pkv_status check_index(const pkv_workspace *ws) {
  if (!ws->seq_lens || !ws->req_pool_indices || !ws->page_table) return PKV_ERR_INVALID;
  if (ws->index_mode == PKV_IDX_FLAT && (!ws->kv_indptr || !ws->kv_indices || ws->max_total_tokens <= 0))
    return PKV_ERR_INVALID;
  return PKV_OK;
}

pkv_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return PKV_OK;
  if (e == cudaErrorNotSupported) return PKV_ERR_UNSUPPORTED;
  return PKV_ERR_CUDA;
}

}  // namespace

extern "C" {

size_t pkv_workspace_bytes(const pkv_workspace *ws, const char *which) {
  if (!ws || !which) return 0;
  const size_t NL = ws->n_layers > 0 ? ws->n_layers : 0;
  const size_t slots = ws->pool_slots > 0 ? ws->pool_slots : 0;
  const size_t hkv = ws->n_kv_heads > 0 ? ws->n_kv_heads : 0;
  const size_t hq = ws->n_q_heads > 0 ? ws->n_q_heads : 0;
  const size_t D = ws->head_dim > 0 ? ws->head_dim : 0;
  const size_t B = ws->max_batch > 0 ? ws->max_batch : 0;
  const size_t S = ws->max_splits > 0 ? ws->max_splits : 0;
  const size_t R = ws->max_reqs > 0 ? ws->max_reqs : 0;
  const size_t MP = ws->max_pages_per_req > 0 ? ws->max_pages_per_req : 0;
  const size_t T = ws->max_total_tokens > 0 ? ws->max_total_tokens : 0;
  if (!strcmp(which, "k_pool") || !strcmp(which, "v_pool")) return NL * slots * hkv * D * 2;
  if (!strcmp(which, "req_pool_indices") || !strcmp(which, "seq_lens") ||
      !strcmp(which, "position_ids") || !strcmp(which, "out_loc"))
    return B * 4;
  if (!strcmp(which, "kv_indptr")) return (B + 1) * 4;
  if (!strcmp(which, "page_table")) return R * MP * 4;
  if (!strcmp(which, "kv_indices")) return T * 4;
  if (!strcmp(which, "o_part")) return B * hq * S * D * 4;
  if (!strcmp(which, "ml_part")) return B * hq * S * 2 * 4;
  if (!strcmp(which, "out")) return B * hq * D * 4;
  if (!strcmp(which, "lse")) return B * hq * 4;
  if (!strcmp(which, "err")) return 4;
  if (!strcmp(which, "split_counters")) return B * hkv * 4;
  if (!strcmp(which, "work_plan")) return plan_bytes();
  return 0;
}

pkv_status pkv_bind_step(const pkv_workspace *ws, int batch, int mode, int layer_begin,
                         int layer_count, const void *k_new, const void *v_new,
                         pkv_stream_t stream) {
  pkv_status st = check_shape(ws);
  if (st != PKV_OK) return st;
  if (mode != PKV_BIND_STEADY && mode != PKV_BIND_REBUILD && mode != PKV_BIND_APPEND_ONLY)
    return PKV_ERR_INVALID;
  if (batch < 0) return PKV_ERR_INVALID;
  if (batch > ws->max_batch || batch > meta_max_batch()) return PKV_ERR_CAPACITY;
  if (layer_count < 0 || layer_begin < 0) return PKV_ERR_INVALID;
  if ((long long)layer_begin + layer_count > ws->n_layers) return PKV_ERR_CAPACITY;
  if (mode != PKV_BIND_APPEND_ONLY) {
    if ((st = check_index(ws)) != PKV_OK) return st;
    if (!ws->position_ids || !ws->kv_indptr || !ws->out_loc) return PKV_ERR_INVALID;
  }
  if (layer_count > 0) {
    if (!ws->k_pool || !ws->v_pool || !ws->out_loc || !k_new || !v_new) return PKV_ERR_INVALID;
    if (!aligned16(ws->k_pool) || !aligned16(ws->v_pool) || !aligned16(k_new) ||
        !aligned16(v_new))
      return PKV_ERR_INVALID;
  }
  if (batch == 0) return PKV_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (mode != PKV_BIND_APPEND_ONLY) {
    if ((st = from_cuda(launch_bind_meta(*ws, batch, mode, s))) != PKV_OK) return st;
    if (ws->index_mode == PKV_IDX_FLAT)
      if ((st = from_cuda(launch_flat_index(*ws, batch, s))) != PKV_OK) return st;
  }
  if (layer_count > 0)
    return from_cuda(launch_append(*ws, batch, layer_begin, layer_count, k_new, v_new, s));
  return PKV_OK;
}

int pkv_choose_splits(const pkv_workspace *ws, int batch, int max_seq_len_hint,
                      long long total_tokens_hint, int num_sms) {
  if (!ws || batch <= 0 || max_seq_len_hint <= 0 || num_sms <= 0 || ws->n_kv_heads <= 0)
    return 1;
  const long long hkv = ws->n_kv_heads, L = max_seq_len_hint;
  const long long total =
      total_tokens_hint > 0 ? total_tokens_hint : (long long)batch * max_seq_len_hint;
  const bool uniform = total * 100 >= (long long)batch * L * 95;
  const long long slots = 2ll * num_sms;  // resident blocks of the tensor-core kernel
  const long long unit_cost = 96;         // per-unit fixed cost, in tokens of streaming
  long long best_t = -1;
  int best_s = 1;
  for (int S = 1; S <= ws->max_splits && S <= 4096; ++S) {
    long long chunk = (L + S - 1) / S;
    chunk = (chunk + 15) / 16 * 16;
    if (S > 1 && chunk < 128) break;
    const long long per_req = (L + chunk - 1) / chunk;
    if (per_req < S) continue;  // same split length as a smaller S
    const long long units = uniform ? (long long)batch * hkv * per_req
                                    : hkv * ((total + chunk - 1) / chunk + batch / 2);
    // uniform lengths: whole waves; mixed lengths (unequal last splits): the
    // fluid share plus half a wave of imbalance.  Fixed point, x1000.
    const long long waves_x1000 =
        uniform ? (units + slots - 1) / slots * 1000 : units * 1000 / slots + 500;
    const long long t = waves_x1000 * (chunk + unit_cost);
    if (best_t < 0 || t < best_t) {
      best_t = t;
      best_s = S;
    }
  }
  return best_s;
}

int pkv_choose_pieces(const pkv_workspace *ws, int batch, int max_seq_len_hint,
                      long long total_tokens_hint, int num_sms) {
  if (!ws || batch <= 0 || max_seq_len_hint <= 0 || num_sms <= 0 || ws->n_kv_heads <= 0 ||
      ws->max_splits < 2)
    return 1;
  const long long L = max_seq_len_hint;
  // Four tiles or fewer: a split saves less streaming than its merge costs.
  if (L <= 256) return 1;
  const long long total = total_tokens_hint > 0 ? total_tokens_hint : (long long)batch * L;
  const long long blocks = 2ll * num_sms;  // resident blocks of the tensor-core kernel
  long long share = (ws->n_kv_heads * total + blocks - 1) / blocks;
  if (share < 128) share = 128;  // two tiles: shorter splits cost more in merging
  const long long S = 3 + (L - 1) / share;
  return (int)(S < ws->max_splits ? S : ws->max_splits);
}

int pkv_choose_extend_splits(const pkv_workspace *ws, int batch, int max_qo_len,
                             int min_seq_len_hint, int num_sms) {
  if (!ws || batch <= 0 || max_qo_len <= 0 || num_sms <= 0 || ws->n_kv_heads <= 0 ||
      ws->n_q_heads <= 0 || ws->n_q_heads % ws->n_kv_heads)
    return 1;
  const int G = ws->n_q_heads / ws->n_kv_heads;
  // the tcgen05 kernel: 128 query rows per CTA, one CTA per SM; the
  // warp-level kernel: 64 rows, two blocks per SM
  const bool umma = extend_umma_supported(*ws);
  const int rows = umma ? 128 : 64;
  const int tq = G <= rows ? rows / G : 1;  // new tokens per block
  const long long units = (long long)((max_qo_len + tq - 1) / tq) * batch * ws->n_kv_heads;
  const long long blocks = (umma ? 1ll : 2ll) * num_sms;
  if (units >= blocks) return 1;
  long long S = blocks / units;
  const long long by_len = min_seq_len_hint > 0 ? min_seq_len_hint / 256 : 1;
  if (by_len < S) S = by_len;
  const long long room = (long long)ws->max_batch * ws->max_splits / ((long long)batch * max_qo_len);
  if (room < S) S = room;
  return (int)(S < 1 ? 1 : S);
}

static pkv_status decode_common(const pkv_workspace *ws, int batch, int layer, const void *q,
                                const void *k_new, const void *v_new, float scale,
                                int num_splits, int flags, int fused, pkv_stream_t stream) {
  pkv_status st = check_shape(ws);
  if (st != PKV_OK) return st;
  if ((st = check_index(ws)) != PKV_OK) return st;
  if (batch < 0 || layer < 0 || num_splits < 1) return PKV_ERR_INVALID;
  if (layer >= ws->n_layers) return PKV_ERR_CAPACITY;
  if (batch > ws->max_batch || num_splits > ws->max_splits) return PKV_ERR_CAPACITY;
  const int G = ws->n_q_heads / ws->n_kv_heads;
  if ((flags & PKV_FLAG_FORCE_SIMT) && (flags & (PKV_FLAG_FORCE_MMA | PKV_FLAG_FORCE_GATHER)))
    return PKV_ERR_INVALID;
  const bool mma_ok = decode_mma_supported(ws->head_dim, G);
  const bool simt_ok = decode_simt_supported(ws->head_dim, G);
  const bool use_mma = (flags & PKV_FLAG_FORCE_MMA) || (mma_ok && !(flags & PKV_FLAG_FORCE_SIMT));
  if (use_mma ? !mma_ok : !simt_ok) return PKV_ERR_UNSUPPORTED;
  if (!q || !ws->k_pool || !ws->v_pool || !ws->out) return PKV_ERR_INVALID;
  if (!aligned16(q) || !aligned16(ws->k_pool) || !aligned16(ws->v_pool) || !aligned16(ws->out))
    return PKV_ERR_INVALID;
  if (num_splits > 1 &&
      (!ws->o_part || !ws->ml_part || !aligned16(ws->o_part) || !aligned8(ws->ml_part)))
    return PKV_ERR_INVALID;
  if ((flags & PKV_FLAG_WRITE_LSE) && !ws->lse) return PKV_ERR_INVALID;
  if ((k_new == nullptr) != (v_new == nullptr)) return PKV_ERR_INVALID;
  if (k_new && (!aligned16(k_new) || !aligned16(v_new) || !ws->out_loc)) return PKV_ERR_INVALID;
  if (fused && num_splits > 1 && !ws->split_counters) return PKV_ERR_INVALID;
  if ((long long)num_splits * batch * ws->n_kv_heads > 0x7fffffffll) return PKV_ERR_CAPACITY;
  if (batch == 0) return PKV_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!use_mma && fused) {
    // The CUDA-core attention has no fused form: run the three steps.
    if (k_new && (st = from_cuda(launch_append(*ws, batch, layer, 1, k_new, v_new, s))) != PKV_OK)
      return st;
    DecodeArgs a{*ws, batch, layer, q, scale, num_splits, flags, nullptr, nullptr, 0, 0};
    if ((st = from_cuda(launch_decode_simt(a, s))) != PKV_OK) return st;
    if (num_splits > 1) return from_cuda(launch_merge(*ws, batch, num_splits, flags, s));
    return PKV_OK;
  }
  DecodeArgs a{*ws, batch, layer, q, scale, num_splits, flags, k_new, v_new, fused, 0};
  return from_cuda(use_mma ? launch_decode_mma(a, s) : launch_decode_simt(a, s));
}

pkv_status pkv_decode_attn(const pkv_workspace *ws, int batch, int layer, const void *q,
                           float scale, int num_splits, int flags, pkv_stream_t stream) {
  return decode_common(ws, batch, layer, q, nullptr, nullptr, scale, num_splits, flags, 0,
                       stream);
}

pkv_status pkv_decode_layer(const pkv_workspace *ws, int batch, int layer, const void *q,
                            const void *k_new, const void *v_new, float scale, int num_splits,
                            int flags, pkv_stream_t stream) {
  return decode_common(ws, batch, layer, q, k_new, v_new, scale, num_splits, flags, 1, stream);
}

pkv_status pkv_plan_step(const pkv_workspace *ws, int batch, int num_splits, int flags,
                         pkv_stream_t stream) {
  pkv_status st = check_shape(ws);
  if (st != PKV_OK) return st;
  if ((st = check_index(ws)) != PKV_OK) return st;
  if (batch < 0 || num_splits < 1) return PKV_ERR_INVALID;
  if (batch > ws->max_batch || num_splits > ws->max_splits) return PKV_ERR_CAPACITY;
  if (!ws->work_plan || !aligned16(ws->work_plan) || !ws->seq_lens) return PKV_ERR_INVALID;
  if ((long long)num_splits * batch * ws->n_kv_heads > 0x7fffffffll) return PKV_ERR_CAPACITY;
  const int G = ws->n_q_heads / ws->n_kv_heads;
  if (batch == 0 || (flags & PKV_FLAG_FORCE_SIMT) || !decode_mma_supported(ws->head_dim, G))
    return PKV_OK;  // no tensor-core launch would read a plan
  DecodeArgs a{*ws, batch, 0, nullptr, 0.f, num_splits, flags, nullptr, nullptr, 1, 0};
  return from_cuda(launch_plan(a, reinterpret_cast<cudaStream_t>(stream)));
}

pkv_status pkv_merge_partials(const pkv_workspace *ws, int batch, int num_splits, int flags,
                              pkv_stream_t stream) {
  pkv_status st = check_shape(ws);
  if (st != PKV_OK) return st;
  if (batch < 0 || num_splits < 1) return PKV_ERR_INVALID;
  if (batch > ws->max_batch || num_splits > ws->max_splits) return PKV_ERR_CAPACITY;
  if (num_splits == 1 || batch == 0) return PKV_OK;
  if (ws->head_dim != 64 && ws->head_dim != 128) return PKV_ERR_UNSUPPORTED;
  if (!ws->o_part || !ws->ml_part || !ws->out) return PKV_ERR_INVALID;
  if (!aligned16(ws->o_part) || !aligned8(ws->ml_part) || !aligned16(ws->out))
    return PKV_ERR_INVALID;
  if ((flags & PKV_FLAG_WRITE_LSE) && !ws->lse) return PKV_ERR_INVALID;
  return from_cuda(launch_merge(*ws, batch, num_splits, flags,
                                reinterpret_cast<cudaStream_t>(stream)));
}

// Checks shared by the two extend calls.
static pkv_status extend_common(const pkv_workspace *ws, int batch, int layer,
                                const int32_t *qo_indptr, int max_qo_len, const void *a,
                                const void *b) {
  pkv_status st = check_shape(ws);
  if (st != PKV_OK) return st;
  if ((st = check_index(ws)) != PKV_OK) return st;
  if (batch < 0 || layer < 0 || max_qo_len < 0) return PKV_ERR_INVALID;
  if (batch > ws->max_batch || layer >= ws->n_layers) return PKV_ERR_CAPACITY;
  if (!extend_supported(ws->head_dim, ws->n_q_heads / ws->n_kv_heads))
    return PKV_ERR_UNSUPPORTED;
  if (!qo_indptr || !a || !b || !ws->k_pool || !ws->v_pool) return PKV_ERR_INVALID;
  if (!aligned16(a) || !aligned16(b) || !aligned16(ws->k_pool) || !aligned16(ws->v_pool))
    return PKV_ERR_INVALID;
  return PKV_OK;
}

pkv_status pkv_extend_attn(const pkv_workspace *ws, int batch, int layer,
                           const int32_t *qo_indptr, int max_qo_len, const void *q, void *out,
                           float scale, int num_splits, int flags, pkv_stream_t stream) {
  pkv_status st = extend_common(ws, batch, layer, qo_indptr, max_qo_len, q, out);
  if (st != PKV_OK) return st;
  if (flags & ~(PKV_FLAG_OUT_F32 | PKV_FLAG_WRITE_LSE | PKV_FLAG_EXTEND_FULL |
                PKV_FLAG_EXTEND_WARP_MMA | PKV_FLAG_PLAN_EARLY))
    return PKV_ERR_INVALID;
  if (num_splits < 1) return PKV_ERR_INVALID;
  // lse[query row, Hq] lives in ws->lse ([max_batch, Hq]): room for every row
  if ((flags & PKV_FLAG_WRITE_LSE) &&
      (!ws->lse || (long long)batch * max_qo_len > ws->max_batch))
    return ws->lse ? PKV_ERR_CAPACITY : PKV_ERR_INVALID;
  if (num_splits > 1) {
    // partials of every (new token, query head, split) in o_part / ml_part
    if (!ws->o_part || !ws->ml_part || !aligned16(ws->o_part) || !aligned8(ws->ml_part))
      return PKV_ERR_INVALID;
    if ((long long)batch * max_qo_len * num_splits > (long long)ws->max_batch * ws->max_splits)
      return PKV_ERR_CAPACITY;
  }
  if ((long long)max_qo_len * num_splits * batch * ws->n_kv_heads > 0x7fffffffll)
    return PKV_ERR_CAPACITY;
  if (batch == 0 || max_qo_len == 0) return PKV_OK;
  return from_cuda(launch_extend(*ws, batch, layer, qo_indptr, max_qo_len, q, out, scale,
                                 num_splits, flags, reinterpret_cast<cudaStream_t>(stream)));
}

pkv_status pkv_extend_append(const pkv_workspace *ws, int batch, int layer,
                             const int32_t *qo_indptr, int max_qo_len, const void *k_new,
                             const void *v_new, pkv_stream_t stream) {
  pkv_status st = extend_common(ws, batch, layer, qo_indptr, max_qo_len, k_new, v_new);
  if (st != PKV_OK) return st;
  if (batch == 0 || max_qo_len == 0) return PKV_OK;
  return from_cuda(launch_extend_append(*ws, batch, layer, qo_indptr, max_qo_len, k_new, v_new,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

pkv_status pkv_merge_lse(int n_rows, int head_dim, const float *o_a, const float *lse_a,
                         const float *o_b, const float *lse_b, void *out, float *lse_out,
                         int flags, pkv_stream_t stream) {
  if (n_rows < 0 || !o_a || !lse_a || !o_b || !lse_b || !out) return PKV_ERR_INVALID;
  if (flags & ~PKV_FLAG_OUT_F32) return PKV_ERR_INVALID;
  if (head_dim <= 0 || head_dim % 64 != 0 || head_dim > 256) return PKV_ERR_UNSUPPORTED;
  if (!aligned16(o_a) || !aligned16(o_b) || !aligned16(out)) return PKV_ERR_INVALID;
  if (n_rows == 0) return PKV_OK;
  return from_cuda(launch_merge_lse(n_rows, head_dim, o_a, lse_a, o_b, lse_b, out, lse_out, flags,
                                    reinterpret_cast<cudaStream_t>(stream)));
}

int pkv_is_steady_increment(const int64_t *prev_ids, const int32_t *prev_lens, int n_prev,
                            const int64_t *ids, const int32_t *lens, int n) {
  if (!prev_ids || !prev_lens || !ids || !lens) return 0;
  if (n <= 0 || n != n_prev) return 0;
  for (int i = 0; i < n; ++i) {
    if (prev_ids[i] != ids[i]) return 0;
    if ((long long)lens[i] != (long long)prev_lens[i] + 1) return 0;
  }
  return 1;
}

const char *pkv_status_string(pkv_status s) {
  switch (s) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported shape";
    case PKV_ERR_CAPACITY: return "beyond workspace capacity";
    case PKV_ERR_CUDA: return "CUDA runtime error";
  }
  return "unknown status";
}

const char *pkv_version(void) { return "pkv 0.1 sm_103a"; }

}  // extern "C"
