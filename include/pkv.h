/*
 * pkv.h -- C ABI of libpkv: batched paged-KV decode attention for GB300 (sm_103a).
 *
 * The engine this follows (AstrAI; its commit-log pages for
 * astrai/inference/core/workspace.py, cache.py and executor.py, cited below as
 * "<file> page, bullet n") runs one decode step as: bind the per-step metadata
 * once (cache.py page, bullets 25, 26, 28), then per layer append the new K/V
 * rows into the 4-D pool (cache.py page, bullets 40-41) and run the split-KV
 * decode kernel whose partial outputs and running max / sum-exp live in
 * caller-owned workspace buffers (workspace.py page, bullets 1, 13-18).
 *
 * Launch overlap: the tensor-core decode kernel is launched with programmatic
 * stream serialization, so it may start while the previous kernel on the
 * stream drains; it waits for that kernel (griddepcontrol.wait) before reading
 * anything another kernel may still be writing, and lets its own successor
 * start only after that wait.
 *
 * Conventions for every entry point
 *  - The library allocates nothing and keeps no data between calls.  Every
 *    buffer is caller-owned device memory at an address that may stay fixed
 *    for the life of the workspace, so a whole step can be captured once into
 *    a CUDA graph and replayed (workspace.py page, bullets 6-7, 17-18).
 *  - Every call is asynchronous on the given stream and never synchronises or
 *    reads device memory on the host.
 *  - Problems the host can see (null pointers, sizes beyond the workspace
 *    capacity, unsupported shapes, misalignment) return a status and launch
 *    nothing.  Problems only the device can see (an out-of-range page id or
 *    slot, a length beyond the table's capacity, a wait that ran out) OR a
 *    bit into the caller's sticky *err word (PKV_DEVERR_*); the affected
 *    outputs are written as an empty result (zeros) and the kernel returns.
 *    No kernel traps, asserts or spins without a limit.
 *  - Element offsets into the pools are computed in 64-bit arithmetic.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL means the legacy default stream. */
typedef struct CUstream_st *pkv_stream_t;

typedef enum pkv_status {
  PKV_OK = 0,
  PKV_ERR_INVALID = 1,     /* null pointer, bad size or mode, misaligned buffer */
  PKV_ERR_UNSUPPORTED = 2, /* head_dim or GQA group size without a kernel     */
  PKV_ERR_CAPACITY = 3,    /* batch / splits / layers beyond the workspace     */
  PKV_ERR_CUDA = 4         /* a CUDA runtime call failed (launch error)        */
} pkv_status;

/* pkv_bind_step modes */
enum {
  PKV_BIND_STEADY = 0,     /* position_ids <- seq_lens; seq_lens += 1; rebuild indptr/out_loc */
  PKV_BIND_REBUILD = 1,    /* take caller-written seq_lens as the new lengths                 */
  PKV_BIND_APPEND_ONLY = 2 /* only copy new K/V rows to pool[layer, out_loc[b]]              */
};

/* pkv_workspace.index_mode */
enum {
  PKV_IDX_PAGE_TABLE = 0,  /* slot(b,t) = page_table[req_pool_indices[b], t/P]*P + t%P */
  PKV_IDX_FLAT = 1         /* P == 1: slot(b,t) = kv_indices[kv_indptr[b] + t]         */
};

/* flags for pkv_decode_attn / pkv_merge_partials */
enum {
  PKV_FLAG_OUT_F32 = 1,    /* write `out` as fp32 instead of bf16 (out must be sized for it) */
  PKV_FLAG_WRITE_LSE = 2,  /* also write lse[b, h] = m + ln(l) (natural log)                */
  PKV_FLAG_FORCE_SIMT = 4, /* use the CUDA-core kernel even where a tensor-core one exists  */
  PKV_FLAG_FORCE_MMA = 8,  /* use the tensor-core kernel (error if the shape has none)      */
  PKV_FLAG_FORCE_GATHER = 16, /* tensor-core kernel: load K/V with cp.async gathers even where
                                 tensor-map TMA boxes apply (P % 16 == 0)                   */
  PKV_FLAG_PLAN_EARLY = 32,  /* tensor-core kernel: the caller guarantees that seq_lens,
                                kv_indptr, kv_indices, req_pool_indices, page_table,
                                out_loc and work_plan were last written at least two
                                launches earlier
                                on this stream (or by the host), so the kernel may read
                                them and start loading K/V before the previous kernel
                                finishes (programmatic dependent launch); q, k_new and
                                all outputs are still touched only after it finishes.
                                pkv_extend_attn (tcgen05 kernel): the same for seq_lens,
                                qo_indptr, req_pool_indices, page_table and the pool
                                rows of each request's cached tokens (those before its
                                new tokens; all of its context with
                                PKV_FLAG_EXTEND_FULL): the CTAs order their units and
                                load those rows early; tiles holding new tokens, q and
                                the outputs wait for the previous kernel.  Either way
                                device error bits may be OR-ed into ws->err before the
                                previous kernel ends, so the operation just before must
                                not be the one that clears it                          */
  PKV_FLAG_FIXED_CHUNK = 64,  /* pkv_decode_layer, tensor-core kernel: cut the KV axis
                                 into pkv_decode_attn's fixed chunks instead of
                                 apportioned splits */
  PKV_FLAG_USE_PLAN = 128,    /* pkv_decode_layer: take the split plan and the first page
                                 ids from ws->work_plan (pkv_plan_step) when it was made
                                 for this batch size, split count and flags; else plan
                                 as without the flag */
  PKV_FLAG_TEST_SKIP_FIRST_TILE = 256, /* test hook, tensor-core kernel: every block's
                                 producer leaves its first tile unloaded, so the bounded
                                 wait for it runs out (~1 s): the launch sets
                                 PKV_DEVERR_TIMEOUT, writes those units empty and
                                 returns, and the context stays usable */
  PKV_FLAG_EXTEND_FULL = 512,  /* pkv_extend_attn: every query row of a request attends all
                                 seq_lens[b] tokens (no causal mask), e.g. a batch's decode
                                 queries over a prefix their requests share */
  PKV_FLAG_EXTEND_WARP_MMA = 1024 /* pkv_extend_attn: the warp-level mma.sync kernel even
                                 where the tcgen05 kernel applies (comparisons) */
};

/* bits OR-ed into *err by device code (sticky; the caller clears the word) */
enum {
  PKV_DEVERR_PAGE = 1,     /* page id < 0 or >= pool_slots / page_size          */
  PKV_DEVERR_LEN = 2,      /* seq_len < 0 or > max_pages_per_req * page_size (or
                              max_seq_len when set)                            */
  PKV_DEVERR_TOTAL = 4,    /* flat mode: kv_indptr[b] + seq_len > max_total_tokens */
  PKV_DEVERR_SLOT = 8,     /* a flat slot or out_loc outside [0, pool_slots)    */
  PKV_DEVERR_TIMEOUT = 16  /* a bounded wait on an async copy ran out (~1 s)    */
};

/*
 * The workspace: shapes plus caller-owned device buffers (the engine's
 * InferenceWorkspace, workspace.py page, bullets 14, 17, 22).  Layouts are
 * dense, row-major, in the element type stated.
 */
typedef struct pkv_workspace {
  int32_t n_layers;          /* NL                                                   */
  int32_t pool_slots;        /* token slots per layer in each pool ("size")          */
  int32_t n_q_heads;         /* Hq                                                   */
  int32_t n_kv_heads;        /* Hkv; Hq % Hkv == 0, G = Hq / Hkv in {1,2,4,8}        */
  int32_t head_dim;          /* D in {64, 128}                                       */
  int32_t page_size;         /* P >= 1 tokens per page; pool_slots % P == 0          */
  int32_t index_mode;        /* PKV_IDX_*                                            */
  int32_t max_batch;         /* capacity of every [B] buffer                         */
  int32_t max_reqs;          /* rows of page_table                                   */
  int32_t max_pages_per_req; /* columns of page_table (tokens per row if P == 1)     */
  int32_t max_splits;        /* S capacity of o_part / ml_part                       */
  int32_t max_total_tokens;  /* capacity of kv_indices (flat mode)                   */

  void *k_pool;              /* bf16 [NL, pool_slots, Hkv, D], 16-byte aligned       */
  void *v_pool;              /* bf16 [NL, pool_slots, Hkv, D], 16-byte aligned       */
  int32_t *req_pool_indices; /* [max_batch]   page_table row of batch entry b        */
  int32_t *page_table;       /* [max_reqs, max_pages_per_req] page ids (slots if P==1) */
  int32_t *seq_lens;         /* [max_batch]   tokens cached incl. the newest; in/out */
  int32_t *position_ids;     /* [max_batch]   0-based position of the newest token   */
  int32_t *kv_indptr;        /* [max_batch+1] exclusive prefix sum of seq_lens       */
  int32_t *out_loc;          /* [max_batch]   slot receiving the newest token        */
  int32_t *kv_indices;       /* [max_total_tokens] flat slots (flat mode only)       */
  float *o_part;             /* >= max_batch*Hq*max_splits*D floats, 16-byte aligned;
                                a call with S splits uses it as dense [batch, Hq, S, D] */
  float *ml_part;            /* >= max_batch*Hq*max_splits*2 floats, 8-byte aligned;
                                used as dense [batch, Hq, S, 2] = (max score, sum exp),
                                ln units                                             */
  void *out;                 /* [max_batch, Hq, D] bf16 (fp32 with PKV_FLAG_OUT_F32) */
  float *lse;                /* [max_batch, Hq] or NULL                               */
  int32_t *err;              /* one sticky int32 of PKV_DEVERR_* bits                */
  int32_t *split_counters;   /* [max_batch * Hkv] zero-initialised once by the caller;
                                used and left at zero by pkv_decode_layer when S > 1;
                                may be NULL if that entry point is not used         */
  int32_t *work_plan;        /* pkv_workspace_bytes(ws, "work_plan") bytes: the step's
                                split plan written by pkv_plan_step and read by
                                pkv_decode_layer with PKV_FLAG_USE_PLAN; may be
                                NULL if those are not used                          */
  int32_t max_seq_len;       /* 0: a request may hold max_pages_per_req * page_size
                                tokens; else at most this many (<= that product), for
                                views whose page_table points part-way into a row of a
                                larger table (the rows keep the stride
                                max_pages_per_req but hold fewer columns).  Longer
                                lengths raise PKV_DEVERR_LEN like any other.  Negative
                                values are PKV_ERR_INVALID                          */
} pkv_workspace;

/*
 * Bytes the named buffer needs for the shapes in `ws` (pointers ignored).
 * `which` is a field name ("k_pool", "o_part", "out" -- sized for fp32 --,
 * ...).  Returns 0 for an unknown name.  Host only; no CUDA call.
 */
size_t pkv_workspace_bytes(const pkv_workspace *ws, const char *which);

/*
 * One per-step metadata bind and/or KV append (cache.py page, bullets 25-28,
 * 40; workspace.py page, bullet 24).
 *   batch        entries 0..batch-1 are live (0 <= batch <= max_batch).
 *   mode         PKV_BIND_STEADY: position_ids[b] = seq_lens[b];
 *                  seq_lens[b] += 1; kv_indptr = [0, cumsum(seq_lens)];
 *                  out_loc[b] = slot(b, seq_lens[b]-1); flat mode also rebuilds
 *                  kv_indices.  All in place, on the device.
 *                PKV_BIND_REBUILD: as STEADY but seq_lens are taken as written
 *                  by the caller (no +1) and position_ids = seq_lens - 1.
 *                PKV_BIND_APPEND_ONLY: no metadata; only the appends below.
 *   layer_begin, layer_count
 *                layers [layer_begin, layer_begin+layer_count) receive the new
 *                rows: K_pool[l, out_loc[b]] = k_new[l-layer_begin, b] (same
 *                for V).  layer_count may be 0 (no append).
 *   k_new, v_new bf16 [layer_count, batch, Hkv, D] device, 16-byte aligned;
 *                may be NULL only when layer_count == 0.
 * Device errors: PKV_DEVERR_PAGE (bad page id for out_loc; out_loc = -1),
 * PKV_DEVERR_LEN, PKV_DEVERR_TOTAL, PKV_DEVERR_SLOT (append skipped).
 */
pkv_status pkv_bind_step(const pkv_workspace *ws, int batch, int mode, int layer_begin,
                         int layer_count, const void *k_new, const void *v_new,
                         pkv_stream_t stream);

/*
 * Split count for a batch, host only.  Work units are (request, KV head,
 * split) and the tensor-core kernel keeps 2 blocks per SM resident, so the
 * time is modelled as waves * (chunk + 96), chunk = ceil(max_seq_len_hint /
 * S) rounded to 16 tokens; the S in [1, max_splits] with the lowest modelled
 * time is returned (splits shorter than 128 tokens are not considered).
 * Near-uniform lengths (total_tokens_hint >= 95% of batch *
 * max_seq_len_hint): units = batch * Hkv * S, waves = ceil(units / (2 *
 * num_sms)).  Otherwise units = Hkv * (ceil(total / chunk) + batch / 2) and
 * waves = units / (2 * num_sms) + 1/2 (unequal last splits).  total_tokens_hint <= 0 means
 * batch * max_seq_len_hint.  Returns 1 for non-positive batch, length or SM
 * count.
 */
int pkv_choose_splits(const pkv_workspace *ws, int batch, int max_seq_len_hint,
                      long long total_tokens_hint, int num_sms);

/*
 * Split cap S for pkv_decode_layer's apportioned splits, host only.  The
 * kernel gives a request of L tokens about L / share splits, share = Hkv *
 * total / blocks over its (up to 2 * num_sms) resident blocks; the value
 * returned leaves headroom over the longest request's share, so a few steps
 * of length growth past the hints do not hit the cap:
 *   share = max(ceil(Hkv * total_tokens_hint / (2 * num_sms)), 128)
 *   S     = min(3 + (max_seq_len_hint - 1) / share, max_splits).
 * total_tokens_hint <= 0 means batch * max_seq_len_hint.  Returns 1 for
 * non-positive batch, length or SM count, for max_splits < 2, and for
 * max_seq_len_hint <= 256 (four 64-token tiles: the merge of a split costs
 * more than the streaming it saves).
 */
int pkv_choose_pieces(const pkv_workspace *ws, int batch, int max_seq_len_hint,
                      long long total_tokens_hint, int num_sms);

/*
 * Split count for pkv_extend_attn, host only.  A block takes R query rows
 * (R / G new tokens of one request and KV head), so a batch has units =
 * ceil(max_qo_len / (R / G)) * batch * Hkv blocks' worth of work; splits of
 * the causal key ranges fill the resident blocks (c per SM) when units fall
 * short of them:
 *   S = 1                                         if units >= c * num_sms,
 *   S = min(c * num_sms / units, min_seq_len_hint / 256)   otherwise,
 * with the geometry of the kernel pkv_extend_attn picks for the workspace:
 * the tcgen05 kernel (page sizes that are a multiple of 16) R = 128, c = 1;
 * the warp-level kernel R = 64, c = 2;
 * so no split is shorter than four 64-key tiles, then at most what the
 * workspace's partials hold (batch * max_qo_len * S <= max_batch * max_splits)
 * and at least 1.  Returns 1 for a null workspace, non-positive batch,
 * max_qo_len or SM count, or a head count G does not divide.
 */
int pkv_choose_extend_splits(const pkv_workspace *ws, int batch, int max_qo_len,
                             int min_seq_len_hint, int num_sms);

/*
 * Split-KV GQA decode attention for one layer (workspace.py page, bullets 1,
 * 14-16).  For every live b and query head h (KV head g = h / G):
 *   s_t = scale * q[b,h,:] . K[layer, slot(b,t), g, :]   for t < seq_lens[b]
 *   o   = sum_t softmax(s)_t V[layer, slot(b,t), g, :]
 *   q           bf16 [batch, Hq, D] device, 16-byte aligned.
 *   scale       softmax scale (fp32), usually 1/sqrt(D).
 *   num_splits  S in [1, max_splits].  The KV axis of every request is cut
 *               into contiguous splits of one common length
 *               chunk = roundup(ceil(max_b seq_lens[b] / S), gran)
 *               (gran = P if P >= 16, else the least multiple of P >= 16),
 *               computed on the device from the live seq_lens.
 *               S == 1: the result goes straight to `out` (and `lse`).
 *               S > 1: split s < n_b = ceil(seq_lens[b] / chunk) of (b,h)
 *               writes o_part[b,h,s,:] (normalised) and ml_part[b,h,s,:] =
 *               (max score, sum exp(s - max)); splits s >= n_b are not
 *               computed (their entries are unspecified) and
 *               pkv_merge_partials reads only the first n_b.
 *   flags       PKV_FLAG_* (OUT_F32 and WRITE_LSE apply when S == 1).
 * Device errors: PKV_DEVERR_PAGE, _LEN, _TOTAL, _SLOT, _TIMEOUT; the affected
 * (b, KV head, split) is written as empty.
 */
pkv_status pkv_decode_attn(const pkv_workspace *ws, int batch, int layer, const void *q,
                           float scale, int num_splits, int flags, pkv_stream_t stream);

/*
 * Log-sum-exp merge of the S split partials into out[b,h,:] (and lse[b,h]
 * with PKV_FLAG_WRITE_LSE):  M = max over non-empty splits of m_s,
 * w_s = l_s exp(m_s - M), out = sum w_s o_s / sum w_s (workspace.py page,
 * bullet 14).  A (b,h) with no non-empty split gets zeros and lse = -inf.
 * num_splits must equal the value given to pkv_decode_attn; with
 * num_splits == 1 this is a no-op returning PKV_OK.
 */
pkv_status pkv_merge_partials(const pkv_workspace *ws, int batch, int num_splits, int flags,
                              pkv_stream_t stream);

/*
 * One layer of a decode step in a single launch: the KV append, split-KV
 * decode attention and the split merge (workspace.py page, bullets 1, 14;
 * cache.py page, bullet 40).  Same results as
 *   pkv_bind_step(PKV_BIND_APPEND_ONLY, layer, 1, k_new, v_new)
 *   pkv_decode_attn(layer, q, scale, num_splits, flags)
 *   pkv_merge_partials(num_splits, flags)
 * after a metadata bind has set seq_lens and out_loc.
 *   k_new, v_new  bf16 [batch, Hkv, D] rows for this layer, or both NULL to
 *                 skip the append.
 *   num_splits    as pkv_decode_attn; with S > 1 ws->split_counters must be
 *                 set (zeroed once; every call leaves it zeroed), and the last
 *                 split to finish for each (request, KV head) merges.
 *                 With S > 1 and batch <= 256 the tensor-core kernel cuts the
 *                 KV axis into apportioned splits instead of fixed chunks: its
 *                 resident blocks are shared out among the requests in
 *                 proportion to their lengths, request b getting n_b splits
 *                 (1 <= n_b <= min(S, ceil(L_b / 128))) of one chunk of its
 *                 own, a multiple of 64 tokens, per KV head, with Hkv * sum n_b
 *                 at most the blocks whenever Hkv * (requests) is; the splits
 *                 are merged as usual (o_part / ml_part slots 0 .. n_b - 1).
 *                 The result equals the fixed-chunk one up to floating-point
 *                 rounding order; PKV_FLAG_FIXED_CHUNK keeps the fixed chunks.
 *   flags         PKV_FLAG_*; with PKV_FLAG_FORCE_SIMT the three steps run as
 *                 separate kernels (the CUDA-core attention has no fusion).
 * Device errors as for pkv_bind_step and pkv_decode_attn.
 */
pkv_status pkv_decode_layer(const pkv_workspace *ws, int batch, int layer, const void *q,
                            const void *k_new, const void *v_new, float scale, int num_splits,
                            int flags, pkv_stream_t stream);

/*
 * The split plan of a step, once for all its layers: what every
 * pkv_decode_layer launch with this batch, num_splits and flags would derive
 * from seq_lens, req_pool_indices / kv_indptr and the page table (usable
 * lengths, index bases, the split length of every request) plus the page ids
 * of each block's first tiles, written to ws->work_plan.  Call it after the
 * step's metadata bind (pkv_bind_step) and before its layers; a layer called
 * with PKV_FLAG_USE_PLAN then reads the plan in one round trip instead of
 * deriving it.  The plan is valid until seq_lens, the request rows, kv_indptr /
 * kv_indices or the page table change (the next bind).  A plan made for other
 * arguments is recognised and ignored.  Nothing is launched (PKV_OK) for
 * batch 0, batch > 256 or shapes without the tensor-core kernel.
 * Device errors: PKV_DEVERR_LEN, PKV_DEVERR_TOTAL.
 */
pkv_status pkv_plan_step(const pkv_workspace *ws, int batch, int num_splits, int flags,
                         pkv_stream_t stream);

/* Size of the device array behind pkv_decode_attn_static_scratch (8 MiB). */
#define PKV_STATIC_SCRATCH_BYTES (8u << 20)

/*
 * pkv_decode_attn followed by pkv_merge_partials, with the split partials
 * kept in a library-owned static device array instead of ws->o_part and
 * ws->ml_part, for callers that cannot allocate device memory (for example a
 * plugin handed only its input and output buffers, or a loop that must not
 * take cudaMalloc's implicit synchronisation).  The pages describe no such
 * entry point; it has no counterpart there.
 *   Arguments and results are those of pkv_decode_attn; ws->o_part and
 *   ws->ml_part are ignored and may be NULL.
 *   Limit: batch * Hq * num_splits * (D + 2) * 4 bytes must fit in
 *   PKV_STATIC_SCRATCH_BYTES, else PKV_ERR_CAPACITY and nothing is launched.
 *   That limit, not ws->max_splits, bounds num_splits here.
 *   The array exists once per GPU that loads the library, for the life of the
 *   process.  The first call on each device looks up its device address
 *   (cudaGetSymbolAddress, with that device current); make that first call
 *   before any stream capture.  No call allocates or frees memory.
 *   All calls share the array and it keeps the last call's contents; calls
 *   whose kernels overlap on the GPU race on it, so issue them in order.
 */
pkv_status pkv_decode_attn_static_scratch(const pkv_workspace *ws, int batch, int layer,
                                          const void *q, float scale, int num_splits,
                                          int flags, pkv_stream_t stream);

/*
 * Paged extend (prefill) attention, the step before decode: each request's
 * newest tokens attend causally over its cached context (the engine keeps
 * the prefill step's qo_indptr in its workspace: workspace.py page, bullet
 * 19; the causal rule is the standard prefill, which the pages do not
 * spell out).
 *   qo_indptr   device int32 [batch + 1]: request b's new tokens are query
 *               rows qo_indptr[b] .. qo_indptr[b + 1] - 1.  They are the last
 *               n_b = qo_indptr[b + 1] - qo_indptr[b] of its seq_lens[b]
 *               tokens, whose K/V are already in the pool (pkv_extend_append);
 *               new token i sits at position p = seq_lens[b] - n_b + i and
 *               attends to positions 0 .. p (query head h reads KV head h / G).
 *   max_qo_len  host upper bound on every n_b (sizes the grid).
 *   q           device bf16 [qo_indptr[batch], Hq, D], 16-byte aligned.
 *   out         device bf16 [qo_indptr[batch], Hq, D] (fp32 with
 *               PKV_FLAG_OUT_F32), 16-byte aligned.
 *   num_splits  S >= 1: every 64-row query block's causal key range
 *               [0, kend) is cut into S splits of ceil(kend / S) keys rounded
 *               up to 64 (later ones may be empty).  S == 1 writes `out`
 *               directly; S > 1 writes the splits' normalised partials and
 *               (max score, sum exp) to ws->o_part / ws->ml_part viewed as
 *               [query row, Hq, S, D] and [query row, Hq, S, 2] (needs
 *               batch * max_qo_len * S <= max_batch * max_splits), then a
 *               second launch merges them into `out` by log-sum-exp.  For
 *               long prefixes with few new tokens, where the unsplit grid has
 *               few blocks.
 *   kernels     page sizes that are a multiple of 16: the tcgen05 kernel (128
 *               query rows per CTA, S = Q K^T and O = P V accumulated in tensor
 *               memory, P applied as bf16 high and low parts); flat indices,
 *               other page sizes or PKV_FLAG_EXTEND_WARP_MMA: the warp-level
 *               mma.sync kernel (64 rows per block).  Both give the same
 *               results up to rounding.
 *   flags       PKV_FLAG_OUT_F32; PKV_FLAG_PLAN_EARLY (see its definition);
 *               PKV_FLAG_WRITE_LSE (also lse[query row * Hq + h] =
 *               max score + ln(sum exp) in ws->lse, which needs batch *
 *               max_qo_len <= max_batch); PKV_FLAG_EXTEND_FULL (no causal
 *               mask: every query row of request b attends all seq_lens[b]
 *               tokens; the rows are then not tokens of the context, so n_b
 *               may exceed seq_lens[b], and seq_lens[b] = 0 gives zero rows
 *               with lse -inf).
 * Reads seq_lens and either req_pool_indices + page_table (page mode) or
 * kv_indptr + kv_indices (flat mode: bind with PKV_BIND_REBUILD first).
 * Host errors: PKV_ERR_INVALID (null pointer, misalignment, batch < 0,
 * max_qo_len < 0, num_splits < 1, another flag), PKV_ERR_CAPACITY (batch >
 * max_batch, layer >= n_layers, the split partials or lse rows do not fit),
 * PKV_ERR_UNSUPPORTED (head_dim not 64 / 128, or G not 1, 2, 4, 8, 16).
 * Device errors: PKV_DEVERR_LEN (n_b < 0, n_b > seq_lens[b] in the causal
 * mode, n_b > max_qo_len, a length out of range, or, with num_splits > 1 or
 * PKV_FLAG_WRITE_LSE, rows past the batch * max_qo_len new tokens the
 * workspace holds (qo_indptr[b + 1] > batch * max_qo_len): that request's
 * rows are not written), PKV_DEVERR_PAGE / _SLOT (a bad index entry: the
 * affected rows are written as zeros), PKV_DEVERR_TIMEOUT.  Nothing is allocated; the call is
 * asynchronous on `stream` and graph-capturable.
 */
pkv_status pkv_extend_attn(const pkv_workspace *ws, int batch, int layer,
                           const int32_t *qo_indptr, int max_qo_len, const void *q, void *out,
                           float scale, int num_splits, int flags, pkv_stream_t stream);

/*
 * Log-sum-exp merge of two attention results over disjoint key sets of the
 * same query rows (a cascade: a prefix the requests share, attended once by
 * pkv_extend_attn with PKV_FLAG_EXTEND_FULL, and each request's own suffix).
 * For each of n_rows rows with normalised outputs o_a, o_b and their lse_a,
 * lse_b (natural log; -inf: no keys):
 *   M = max(lse_a, lse_b), w = exp(lse - M),
 *   out = (w_a o_a + w_b o_b) / (w_a + w_b)   (zeros when both are -inf)
 * and lse_out = M + ln(w_a + w_b) when lse_out is not NULL.
 *   o_a, o_b   device fp32 [n_rows, head_dim], 16-byte aligned.
 *   out        device bf16 [n_rows, head_dim] (fp32 with PKV_FLAG_OUT_F32).
 * head_dim: a multiple of 64, at most 256.  Host errors: PKV_ERR_INVALID
 * (null pointer, misalignment, n_rows < 0, other flags), PKV_ERR_UNSUPPORTED
 * (head_dim).  Asynchronous on `stream`.
 */
pkv_status pkv_merge_lse(int n_rows, int head_dim, const float *o_a, const float *lse_a,
                         const float *o_b, const float *lse_b, void *out, float *lse_out,
                         int flags, pkv_stream_t stream);

/*
 * Extend append: the new tokens' K and V rows into the pool.  k_new, v_new:
 * device bf16 [qo_indptr[batch], Hkv, D], 16-byte aligned; row
 * qo_indptr[b] + i goes to layer `layer`, slot of position
 * seq_lens[b] - n_b + i (page-table walk, or kv_indices in flat mode).
 * Same request checks as pkv_extend_attn (PKV_DEVERR_LEN: the request is
 * skipped); a bad page id or slot raises PKV_DEVERR_PAGE / _SLOT and that
 * row is skipped.  Host errors as pkv_extend_attn.
 */
pkv_status pkv_extend_append(const pkv_workspace *ws, int batch, int layer,
                             const int32_t *qo_indptr, int max_qo_len, const void *k_new,
                             const void *v_new, pkv_stream_t stream);

/*
 * Host steady-state test (cache.py page, bullets 1-4): non-zero when the
 * task ids are the same, in the same order, as at the last bind and every
 * length grew by exactly one, so a PKV_BIND_STEADY step is valid; zero means
 * the caller must write seq_lens and bind with PKV_BIND_REBUILD.
 * Host arrays; n_prev / n may differ (then the result is 0).
 */
int pkv_is_steady_increment(const int64_t *prev_ids, const int32_t *prev_lens, int n_prev,
                            const int64_t *ids, const int32_t *lens, int n);

/* Static string for a status code. */
const char *pkv_status_string(pkv_status status);

/* Library version, e.g. "pkv 0.1 sm_103a". */
const char *pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
