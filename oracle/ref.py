"""Plain, slow, fp64 reference for the paged-KV decode path.

TEST INFRASTRUCTURE ONLY -- never imported by the product package.

Sources (the engine's commit-log pages, AstrAI by ViperEkura; cited as
"<page> page, bullet n", bullets counted from the top of each page):
  * workspace.py page  -- commit 0b661ba, astrai/inference/core/workspace.py
  * cache.py page      -- commit cbc5844, astrai/inference/core/cache.py
  * executor.py page   -- commit e0f7fa8, astrai/inference/core/executor.py

Readings taken where the pages are silent:
  * query head h reads KV head h // G, G = Hq / Hkv (contiguous groups);
  * the new token is appended before attention, so it is attended;
  * a steady step sets position_ids to the old length, then adds 1 to
    seq_lens; kv_indptr counts tokens (exclusive prefix sum of seq_lens);
  * page mode: token t of request b lives in slot
    page_table[req_pool_indices[b], t // P] * P + t % P;
    flat mode (P = 1): slot kv_indices[kv_indptr[b] + t], where kv_indices is
    the concatenation of each request's row of the request-to-token table;
  * split partials hold the normalised partial output and (m, l) in natural
    log units; splits are contiguous token ranges of one common length that
    is a multiple of the split granularity; an empty split has m = -inf,
    l = 0 and is skipped by the merge;
  * extend (prefill) attention is causal: a request's n new tokens are the
    last n of its context and each attends to its own position and earlier.

Everything is written out as loops over requests, heads and tokens; numpy
only supplies elementwise exp / log, sums and dot products.
"""
from __future__ import annotations

import math

import numpy as np

PAGE_TABLE = 0
FLAT = 1

STEADY = 0
REBUILD = 1


# ---------------------------------------------------------------------------
# bf16 handling (exact): a bf16 value is the top half of an IEEE fp32.
# ---------------------------------------------------------------------------

def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact fp64 values of bf16 numbers given as their 16-bit patterns."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def tensor_bits(t) -> np.ndarray:
    """16-bit patterns of a torch bf16 CPU tensor, as a numpy uint16 array."""
    import torch  # local: the oracle only needs torch to read its inputs
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------------------
# Metadata (cache.py page, bullets 25, 26, 28; workspace.py page, bullet 24)
# ---------------------------------------------------------------------------

def slot_of_token(b, t, *, page_table, req_pool_indices, page_size):
    """Physical slot of logical token t of batch entry b (page-table walk).

    The 4-D storage is indexed by (layer, slot) (cache.py page, bullets 40,
    41); the request-to-token table row is selected by req_pool_indices
    (cache.py page, bullet 26)."""
    row = int(req_pool_indices[b])
    page = int(page_table[row][t // page_size])
    return page * page_size + t % page_size


def bind(seq_lens, *, req_pool_indices, page_table, page_size, mode, index_mode=PAGE_TABLE):
    """Per-step decode metadata.

    STEADY: position_ids <- old seq_lens; seq_lens <- seq_lens + 1
    (cache.py page, bullets 25-26).  REBUILD: lengths taken as given,
    position_ids = seq_lens - 1.  In both, kv_indptr is the exclusive prefix
    sum of the new seq_lens, computed once per step (cache.py page, bullet
    28), and out_loc[b] is the slot of the newest token.  Flat mode also
    builds kv_indices, the concatenated per-request token slots.
    Returns a dict of python int lists.
    """
    B = len(seq_lens)
    old = [int(x) for x in seq_lens]
    if mode == STEADY:
        new = [x + 1 for x in old]
        pos = list(old)
    elif mode == REBUILD:
        new = list(old)
        pos = [x - 1 for x in old]
    else:
        raise ValueError(mode)
    indptr = [0]
    for b in range(B):
        indptr.append(indptr[-1] + new[b])
    out_loc = []
    for b in range(B):
        if new[b] >= 1:
            out_loc.append(slot_of_token(b, new[b] - 1, page_table=page_table,
                                         req_pool_indices=req_pool_indices,
                                         page_size=page_size))
        else:
            out_loc.append(-1)
    res = {"seq_lens": new, "position_ids": pos, "kv_indptr": indptr, "out_loc": out_loc}
    if index_mode == FLAT:
        flat = []
        for b in range(B):
            for t in range(new[b]):
                flat.append(slot_of_token(b, t, page_table=page_table,
                                          req_pool_indices=req_pool_indices, page_size=1))
        res["kv_indices"] = flat
    return res


def token_slots(b, seq_len, *, page_table=None, req_pool_indices=None, page_size=1,
                index_mode=PAGE_TABLE, kv_indptr=None, kv_indices=None):
    """Slots of tokens 0..seq_len-1 of entry b, walking the index structure."""
    if index_mode == FLAT:
        base = int(kv_indptr[b])
        return [int(kv_indices[base + t]) for t in range(seq_len)]
    return [slot_of_token(b, t, page_table=page_table, req_pool_indices=req_pool_indices,
                          page_size=page_size) for t in range(seq_len)]


def append_rows(pool_bits, layer, out_loc, new_bits):
    """KV append: pool[layer, out_loc[b]] <- new[b] (cache.py page, bullet 40).

    Works on 16-bit patterns, so it is exact; returns a modified copy."""
    out = np.array(pool_bits, copy=True)
    for b, loc in enumerate(out_loc):
        out[layer, int(loc)] = new_bits[b]
    return out


# ---------------------------------------------------------------------------
# Attention (workspace.py page, bullets 1 and 14: the decode kernel and its
# split partial buffers).
# ---------------------------------------------------------------------------

def kv_head_of(h, n_q_heads, n_kv_heads):
    """GQA map (reading): contiguous groups of G = Hq / Hkv query heads."""
    return h // (n_q_heads // n_kv_heads)


def attend(q, K, V, scale):
    """softmax(scale * K q) . V for one query vector.

    q: (D,), K, V: (L, D) float64.  Returns (o (D,), lse).  L = 0 gives
    o = 0, lse = -inf."""
    L = K.shape[0]
    if L == 0:
        return np.zeros(V.shape[1]), -math.inf
    s = np.empty(L)
    for t in range(L):
        s[t] = scale * float(np.dot(K[t], q))
    m = float(np.max(s))
    e = np.exp(s - m)
    z = float(np.sum(e))
    o = (e @ V) / z
    return o, m + math.log(z)


def decode_attention(q_bits, k_pool_bits, v_pool_bits, layer, slots_per_req, scale,
                     n_kv_heads, heads=None):
    """Decode attention for every (b, h), gathering K/V through the slots.

    q_bits: uint16 (B, Hq, D); pools: uint16 (NL, slots, Hkv, D);
    slots_per_req[b]: list of physical slots of tokens 0..L_b-1.
    ``scale`` is taken as the exact fp64 value of the fp32 number passed.
    ``heads``: optional list of (b, h) to compute (others stay 0).
    Returns o (B, Hq, D) float64 and lse (B, Hq)."""
    q = bf16_bits_to_f64(q_bits)
    B, Hq, D = q.shape
    scale = float(np.float32(scale))
    o = np.zeros((B, Hq, D))
    lse = np.full((B, Hq), -math.inf)
    want = heads if heads is not None else [(b, h) for b in range(B) for h in range(Hq)]
    cache = {}
    for b, h in want:
        g = kv_head_of(h, Hq, n_kv_heads)
        key = (b, g)
        if key not in cache:
            sl = np.asarray(slots_per_req[b], dtype=np.int64)
            K = bf16_bits_to_f64(k_pool_bits[layer, sl, g]) if sl.size else np.zeros((0, D))
            V = bf16_bits_to_f64(v_pool_bits[layer, sl, g]) if sl.size else np.zeros((0, D))
            cache = {key: (K, V)}
        K, V = cache[key]
        o[b, h], lse[b, h] = attend(q[b, h], K, V, scale)
    return o, lse


# ---------------------------------------------------------------------------
# Split-KV partials and their merge (workspace.py page, bullet 14).
# ---------------------------------------------------------------------------

def split_granularity(page_size):
    """Split lengths are multiples of this: the page size when a page holds
    at least 16 tokens, else the smallest multiple of the page size >= 16."""
    return page_size if page_size >= 16 else page_size * (-(-16 // page_size))


def split_chunk(seq_lens, num_splits, page_size):
    """Common split length for a batch: ceil(max L / S) rounded up to the
    split granularity, so no request needs more than S splits."""
    gran = split_granularity(page_size)
    mx = max([int(x) for x in seq_lens] + [1])
    c = -(-mx // int(num_splits))
    return -(-c // gran) * gran


def partial(q, K, V, scale):
    """(m, l, o) of one split: m = max score, l = sum exp(s - m),
    o = normalised partial output.  Empty split: (-inf, 0, 0)."""
    L = K.shape[0]
    if L == 0:
        return -math.inf, 0.0, np.zeros(V.shape[1])
    s = np.array([scale * float(np.dot(K[t], q)) for t in range(L)])
    m = float(np.max(s))
    e = np.exp(s - m)
    l = float(np.sum(e))
    return m, l, (e @ V) / l


def merge(ms, ls, os_):
    """Log-sum-exp merge of split partials.

    M = max over non-empty splits of m_s; w_s = l_s exp(m_s - M);
    out = sum_s w_s o_s / sum_s w_s; lse = M + log sum_s w_s.
    All splits empty: out = 0, lse = -inf."""
    live = [s for s in range(len(ms)) if ls[s] > 0]
    if not live:
        return np.zeros(np.asarray(os_[0]).shape), -math.inf
    M = max(ms[s] for s in live)
    num = 0.0
    den = 0.0
    for s in live:
        w = ls[s] * math.exp(ms[s] - M)
        num = num + w * np.asarray(os_[s], dtype=np.float64)
        den += w
    return num / den, M + math.log(den)


def split_partials(q_bits, k_pool_bits, v_pool_bits, layer, slots_per_req, scale,
                   n_kv_heads, num_splits, page_size, seq_lens, heads=None):
    """Per-split partials in the layout of the decode split buffers.

    Returns o_part (B, Hq, S, D) and ml_part (B, Hq, S, 2) float64; split s of
    request b covers tokens [s*chunk, min((s+1)*chunk, L_b))."""
    q = bf16_bits_to_f64(q_bits)
    B, Hq, D = q.shape
    S = int(num_splits)
    scale = float(np.float32(scale))
    chunk = split_chunk(seq_lens, S, page_size)
    o_part = np.zeros((B, Hq, S, D))
    ml = np.zeros((B, Hq, S, 2))
    ml[..., 0] = -math.inf
    want = heads if heads is not None else [(b, h) for b in range(B) for h in range(Hq)]
    for b, h in want:
        g = kv_head_of(h, Hq, n_kv_heads)
        L = int(seq_lens[b])
        sl = np.asarray(slots_per_req[b], dtype=np.int64)
        for s in range(S):
            lo, hi = s * chunk, min((s + 1) * chunk, L)
            if lo >= hi:
                continue
            K = bf16_bits_to_f64(k_pool_bits[layer, sl[lo:hi], g])
            V = bf16_bits_to_f64(v_pool_bits[layer, sl[lo:hi], g])
            m, l, o = partial(q[b, h], K, V, scale)
            o_part[b, h, s] = o
            ml[b, h, s] = (m, l)
    return o_part, ml


def merge_partials(o_part, ml_part):
    """Merge (B, Hq, S, D) partials into (B, Hq, D) outputs and (B, Hq) lse."""
    B, Hq, S, D = o_part.shape
    out = np.zeros((B, Hq, D))
    lse = np.full((B, Hq), -math.inf)
    for b in range(B):
        for h in range(Hq):
            out[b, h], lse[b, h] = merge(list(ml_part[b, h, :, 0]), list(ml_part[b, h, :, 1]),
                                         list(o_part[b, h]))
    return out, lse


# ---------------------------------------------------------------------------
# Extend (prefill) attention: the step before decode, whose per-request query
# offsets qo_indptr the workspace holds (workspace.py page, bullet 19).  The
# pages give no formula; reading: the standard causal prefill.  Request b holds
# L_b tokens in the pool, the last n_b of them new; new token i sits at
# position L_b - n_b + i and attends tokens 0 .. L_b - n_b + i.
# ---------------------------------------------------------------------------

def extend_positions(seq_len, n_new):
    """Positions of a request's n_new newest tokens in its context of
    seq_len tokens."""
    return [seq_len - n_new + i for i in range(n_new)]


def extend_attention(q_bits, k_pool_bits, v_pool_bits, layer, slots_per_req, qo_lens, scale,
                     n_kv_heads, rows=None):
    """Causal attention of each request's new tokens over its context.

    q_bits: uint16 (sum n_b, Hq, D), the new tokens' queries in request
    order; slots_per_req[b]: physical slots of tokens 0..L_b-1 (new ones
    included); qo_lens[b] = n_b.  ``rows``: optional list of (query row, h)
    to compute (others stay 0).  Returns o (sum n_b, Hq, D) float64 and lse
    (sum n_b, Hq)."""
    q = bf16_bits_to_f64(q_bits)
    T, Hq, D = q.shape
    scale = float(np.float32(scale))
    o = np.zeros((T, Hq, D))
    lse = np.full((T, Hq), -math.inf)
    owner = []  # query row -> (request, position)
    for b, n in enumerate(qo_lens):
        for pos in extend_positions(len(slots_per_req[b]), int(n)):
            owner.append((b, pos))
    assert len(owner) == T, "q rows do not match the new-token counts"
    want = rows if rows is not None else [(r, h) for r in range(T) for h in range(Hq)]
    for r, h in want:
        b, pos = owner[r]
        g = kv_head_of(h, Hq, n_kv_heads)
        sl = np.asarray(slots_per_req[b][:pos + 1], dtype=np.int64)
        K = bf16_bits_to_f64(k_pool_bits[layer, sl, g]) if sl.size else np.zeros((0, D))
        V = bf16_bits_to_f64(v_pool_bits[layer, sl, g]) if sl.size else np.zeros((0, D))
        o[r, h], lse[r, h] = attend(q[r, h], K, V, scale)
    return o, lse


def extend_append(pool_bits, layer, slots_per_req, qo_lens, new_bits):
    """Extend append: the new tokens' rows (new_bits (sum n_b, Hkv, D), in
    request order) go to the slots of the last n_b positions of each request."""
    out = pool_bits.copy()
    r = 0
    for b, n in enumerate(qo_lens):
        for pos in extend_positions(len(slots_per_req[b]), int(n)):
            out[layer, slots_per_req[b][pos]] = new_bits[r]
            r += 1
    return out


# ---------------------------------------------------------------------------
# Host-side steady-state test (cache.py page, bullets 1-4).
# ---------------------------------------------------------------------------

def is_steady_increment(prev_ids, prev_lens, ids, lens):
    """True when the task set and order are unchanged and every length grew
    by exactly one since the last bind; otherwise metadata is rebuilt."""
    if prev_ids is None or len(prev_ids) != len(ids) or len(ids) == 0:
        return False
    for a, b in zip(prev_ids, ids):
        if int(a) != int(b):
            return False
    for a, b in zip(prev_lens, lens):
        if int(b) != int(a) + 1:
            return False
    return True
