"""Pins for the CPU fp64 oracle (no GPU).

Each ``pin_*`` checks the oracle against something other than itself: a
hand-worked example from ``tests/golden/``, a closed form, an invariant, or
the float64 library routine ``scaled_dot_product_attention`` (which the oracle
never calls).  ``test_planted_mistakes`` re-runs the pins against deliberately
broken copies of oracle functions and requires each break to be caught.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle.ref as R
import pkv_inputs as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _num(x):
    if isinstance(x, str):
        if "/" in x:
            a, b = x.split("/")
            return float(a) / float(b)
        return {"ln2": math.log(2), "ln3": math.log(3), "ln4": math.log(4), "ln7": math.log(7),
                "-inf": -math.inf}[x]
    return float(x)


def _arr(a):
    return np.array([[_num(v) for v in row] if isinstance(row, list) else _num(row) for row in a],
                    dtype=np.float64)


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bits(x):
    """bf16 bit patterns of fp64 values that are exactly representable."""
    t = torch.tensor(np.asarray(x, dtype=np.float64)).to(torch.bfloat16)
    assert torch.equal(t.to(torch.float64), torch.tensor(np.asarray(x, dtype=np.float64))), \
        "fixture value not bf16-exact"
    return R.tensor_bits(t)


def _tiny_problem(seed=7, B=3, Hq=4, Hkv=2, D=8, P=4, lens=(5, 1, 11), NL=2, layer=1):
    p = W.make_problem("tiny", batch=B, n_layers=NL, n_q_heads=Hq, n_kv_heads=Hkv,
                       head_dim=D, page_size=P, seq_lens=list(lens), seed=seed)
    q = W.normal_bf16((B, Hq, D), seed + 100)
    slots = [R.token_slots(b, int(p.seq_lens[b]), page_table=p.page_table.numpy(),
                           req_pool_indices=p.req_pool_indices.numpy(), page_size=P)
             for b in range(B)]
    return p, q, slots, layer


# ------------------------------------------------------------------ pins ---

def pin_golden_attend():
    for name in ("attend_two_tokens.json", "attend_three_tokens_scale.json"):
        g = _load(name)
        o, lse = R.attend(_arr(g["q"]), _arr(g["K"]), _arr(g["V"]), _num(g["scale"]))
        assert np.allclose(o, _arr(g["o"]), rtol=0, atol=1e-13), (name, o)
        assert abs(lse - _num(g["lse"])) < 1e-13, (name, lse)


def pin_golden_gqa_map():
    g = _load("gqa_map.json")
    Hq, Hkv, D = g["n_q_heads"], g["n_kv_heads"], g["head_dim"]
    V = np.array(g["V_slot_head"], dtype=np.float64)[None, :, :, None]  # (1, slots, Hkv, 1)
    vb = _bits(V)
    kb = _bits(np.zeros_like(V))
    qb = _bits(np.zeros((1, Hq, D)))
    slots = [R.token_slots(0, g["seq_len"], page_table=g["page_table"],
                           req_pool_indices=g["req_pool_indices"], page_size=g["page_size"])]
    o, _ = R.decode_attention(qb, kb, vb, 0, slots, 0.5, Hkv)
    assert np.allclose(o[0, :, 0], g["o"], rtol=0, atol=1e-13), o[0, :, 0]


def pin_golden_bind():
    for name in ("bind_steady_paged.json", "bind_rebuild_flat.json"):
        g = _load(name)
        mode = R.STEADY if g["mode"] == "steady" else R.REBUILD
        flat = R.FLAT if g["page_size"] == 1 and "kv_indices" in g["expect"] else R.PAGE_TABLE
        res = R.bind(g["seq_lens"], req_pool_indices=g["req_pool_indices"],
                     page_table=g["page_table"], page_size=g["page_size"], mode=mode,
                     index_mode=flat)
        for k, v in g["expect"].items():
            assert res[k] == v, (name, k, res[k], v)


def pin_golden_merge():
    g = _load("merge_two_splits.json")
    out, lse = R.merge([_num(x) for x in g["m"]], [_num(x) for x in g["l"]],
                       [np.array(o) for o in g["o"]])
    assert np.allclose(out, g["out"], rtol=0, atol=1e-14), out
    assert abs(lse - _num(g["lse"])) < 1e-14


def pin_single_token_is_v():
    # One cached token: the softmax weight is exactly 1, so o equals that V row.
    p, q, _, layer = _tiny_problem(lens=(1, 1, 1))
    slots = [R.token_slots(b, 1, page_table=p.page_table.numpy(),
                           req_pool_indices=p.req_pool_indices.numpy(), page_size=p.page_size)
             for b in range(p.batch)]
    kb, vb = R.tensor_bits(p.k_pool), R.tensor_bits(p.v_pool)
    o, lse = R.decode_attention(R.tensor_bits(q), kb, vb, layer, slots, p.scale, p.n_kv_heads)
    for b in range(p.batch):
        for h in range(p.n_q_heads):
            v = R.bf16_bits_to_f64(vb[layer, slots[b][0], h // p.group])
            assert np.array_equal(o[b, h], v), (b, h)


def pin_uniform_cases_give_mean_v():
    # Identical keys, q = 0 and scale = 0 each make every score equal, so the
    # output is the plain mean of the request's V rows.
    p, q, slots, layer = _tiny_problem()
    kb, vb = R.tensor_bits(p.k_pool).copy(), R.tensor_bits(p.v_pool)
    qb = R.tensor_bits(q)
    for case in ("same_keys", "q0", "scale0"):
        k_use, q_use, sc = kb, qb, p.scale
        if case == "same_keys":
            k_use = kb.copy()
            for b in range(p.batch):
                for t, s in enumerate(slots[b]):
                    k_use[layer, s] = kb[layer, slots[b][0]]
        elif case == "q0":
            q_use = np.zeros_like(qb)
        else:
            sc = 0.0
        o, _ = R.decode_attention(q_use, k_use, vb, layer, slots, sc, p.n_kv_heads)
        for b in range(p.batch):
            for h in range(p.n_q_heads):
                V = R.bf16_bits_to_f64(vb[layer, np.array(slots[b]), h // p.group])
                assert np.allclose(o[b, h], V.mean(axis=0), rtol=0, atol=1e-12), (case, b, h)


def pin_matches_sdpa_f64():
    # Library special case: dense SDPA in float64 with grouped KV heads on the
    # contiguous (unpaged) per-request K/V.
    p, q, slots, layer = _tiny_problem(lens=(5, 2, 13))
    kb, vb, qb = R.tensor_bits(p.k_pool), R.tensor_bits(p.v_pool), R.tensor_bits(q)
    o, lse = R.decode_attention(qb, kb, vb, layer, slots, p.scale, p.n_kv_heads)
    kf = p.k_pool.to(torch.float64)
    vf = p.v_pool.to(torch.float64)
    qf = q.to(torch.float64)
    for b in range(p.batch):
        idx = torch.tensor(slots[b])
        K = kf[layer, idx].permute(1, 0, 2)[None]  # (1, Hkv, L, D)
        V = vf[layer, idx].permute(1, 0, 2)[None]
        Q = qf[b][None, :, None, :]                # (1, Hq, 1, D)
        ref = torch.nn.functional.scaled_dot_product_attention(
            Q, K, V, scale=float(np.float32(p.scale)), enable_gqa=True)[0, :, 0]
        assert np.allclose(o[b], ref.numpy(), rtol=0, atol=1e-12), b
        s = torch.einsum("hd,hld->hl", qf[b], K[0].repeat_interleave(p.group, 0))
        s = s * float(np.float32(p.scale))
        assert np.allclose(lse[b], torch.logsumexp(s, -1).numpy(), rtol=0, atol=1e-12)


def pin_page_shuffle_invariance():
    # Moving physical pages (data and table entries together) leaves the
    # output bit-identical.
    p, q, slots, layer = _tiny_problem()
    kb, vb, qb = R.tensor_bits(p.k_pool), R.tensor_bits(p.v_pool), R.tensor_bits(q)
    o1, l1 = R.decode_attention(qb, kb, vb, layer, slots, p.scale, p.n_kv_heads)
    P = p.page_size
    n_pages = p.pool_slots // P
    perm = np.random.default_rng(3).permutation(n_pages)  # new_page = perm[old_page]
    k2, v2 = np.empty_like(kb), np.empty_like(vb)
    for old in range(n_pages):
        k2[:, perm[old] * P:(perm[old] + 1) * P] = kb[:, old * P:(old + 1) * P]
        v2[:, perm[old] * P:(perm[old] + 1) * P] = vb[:, old * P:(old + 1) * P]
    table = p.page_table.numpy().copy()
    table[table >= 0] = perm[table[table >= 0]]
    slots2 = [R.token_slots(b, int(p.seq_lens[b]), page_table=table,
                            req_pool_indices=p.req_pool_indices.numpy(), page_size=P)
              for b in range(p.batch)]
    o2, l2 = R.decode_attention(qb, k2, v2, layer, slots2, p.scale, p.n_kv_heads)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def pin_batch_permutation():
    # Reordering the batch reorders the outputs and nothing else.
    p, q, slots, layer = _tiny_problem()
    kb, vb, qb = R.tensor_bits(p.k_pool), R.tensor_bits(p.v_pool), R.tensor_bits(q)
    o1, _ = R.decode_attention(qb, kb, vb, layer, slots, p.scale, p.n_kv_heads)
    order = [2, 0, 1]
    o2, _ = R.decode_attention(qb[order], kb, vb, layer, [slots[i] for i in order], p.scale,
                               p.n_kv_heads)
    assert np.array_equal(o1[order], o2)


def pin_mha_reduces():
    # G = 1: every query head reads its own KV head; compare with SDPA without GQA.
    p, q, slots, layer = _tiny_problem(Hq=2, Hkv=2)
    kb, vb, qb = R.tensor_bits(p.k_pool), R.tensor_bits(p.v_pool), R.tensor_bits(q)
    o, _ = R.decode_attention(qb, kb, vb, layer, slots, p.scale, p.n_kv_heads)
    for b in range(p.batch):
        idx = torch.tensor(slots[b])
        K = p.k_pool.to(torch.float64)[layer, idx].permute(1, 0, 2)[None]
        V = p.v_pool.to(torch.float64)[layer, idx].permute(1, 0, 2)[None]
        Q = q.to(torch.float64)[b][None, :, None, :]
        ref = torch.nn.functional.scaled_dot_product_attention(
            Q, K, V, scale=float(np.float32(p.scale)))[0, :, 0]
        assert np.allclose(o[b], ref.numpy(), rtol=0, atol=1e-12)


def pin_split_merge_identity():
    # The log-sum-exp merge of any contiguous partition (empty parts allowed)
    # reproduces unsplit attention.
    rng = np.random.default_rng(11)
    for trial in range(20):
        L = int(rng.integers(1, 40))
        D = 6
        q = rng.standard_normal(D) * 2
        K = rng.standard_normal((L, D)) * 2
        V = rng.standard_normal((L, D))
        o, lse = R.attend(q, K, V, 0.7)
        cuts = sorted(rng.integers(0, L + 1, size=int(rng.integers(0, 5))).tolist())
        edges = [0] + cuts + [L]
        ms, ls, os_ = [], [], []
        for a, b in zip(edges[:-1], edges[1:]):
            m, l, op = R.partial(q, K[a:b], V[a:b], 0.7)
            ms.append(m), ls.append(l), os_.append(op)
        out, lse2 = R.merge(ms, ls, os_)
        assert np.allclose(out, o, rtol=0, atol=1e-12), trial
        assert abs(lse2 - lse) < 1e-12


def pin_split_partials_layout():
    # Split partials over the batch's common chunk merge back to attention,
    # and every split past a request's length is empty.
    p, q, slots, layer = _tiny_problem(lens=(5, 1, 23), P=4)
    kb, vb, qb = R.tensor_bits(p.k_pool), R.tensor_bits(p.v_pool), R.tensor_bits(q)
    o, lse = R.decode_attention(qb, kb, vb, layer, slots, p.scale, p.n_kv_heads)
    for S in (1, 2, 3, 8):
        op, ml = R.split_partials(qb, kb, vb, layer, slots, p.scale, p.n_kv_heads, S,
                                  p.page_size, p.seq_lens.tolist())
        chunk = R.split_chunk(p.seq_lens.tolist(), S, p.page_size)
        for b in range(p.batch):
            n = -(-int(p.seq_lens[b]) // chunk)
            assert n <= S
            assert np.all(ml[b, :, n:, 1] == 0) and np.all(np.isneginf(ml[b, :, n:, 0]))
        out, lse2 = R.merge_partials(op, ml)
        assert np.allclose(out, o, rtol=0, atol=1e-12), S
        assert np.allclose(lse2, lse, rtol=0, atol=1e-12)


def pin_split_chunk():
    for lens in ([1], [17, 3], [8192, 5, 100], [65536]):
        for S in (1, 2, 7, 64):
            for P in (1, 4, 16, 32):
                c = R.split_chunk(lens, S, P)
                gran = P if P >= 16 else 16 if 16 % P == 0 else P * math.ceil(16 / P)
                assert c % gran == 0 and c * S >= max(lens)
                assert (c - gran) * S < max(lens) or c == gran


def pin_bind_closed_form():
    # After k steady steps: seq_lens = L0 + k, position_ids = seq_lens - 1,
    # kv_indptr[b] = kv_indptr0[b] + k*b, out_loc = slot of token L0 + k - 1.
    p = W.make_problem("t", batch=5, n_layers=1, n_q_heads=2, n_kv_heads=1, head_dim=8,
                       page_size=4, seq_lens=[3, 9, 1, 4, 16], steps=12, seed=5)
    tab, rows = p.page_table.numpy(), p.req_pool_indices.numpy()
    L0 = p.seq_lens.tolist()
    base = R.bind(L0, req_pool_indices=rows, page_table=tab, page_size=4, mode=R.REBUILD)
    lens = L0
    for k in range(1, 13):
        res = R.bind(lens, req_pool_indices=rows, page_table=tab, page_size=4, mode=R.STEADY)
        lens = res["seq_lens"]
        assert lens == [x + k for x in L0]
        assert res["position_ids"] == [x - 1 for x in lens]
        assert res["kv_indptr"] == [base["kv_indptr"][b] + k * b for b in range(6)]
        for b in range(5):
            t = L0[b] + k - 1
            row = rows[b]
            assert res["out_loc"][b] == tab[row, t // 4] * 4 + t % 4


def pin_append():
    rng = np.random.default_rng(2)
    pool = rng.integers(0, 65535, size=(3, 10, 2, 4)).astype(np.uint16)
    new = rng.integers(0, 65535, size=(2, 2, 4)).astype(np.uint16)
    out = R.append_rows(pool, 1, [7, 2], new)
    assert np.array_equal(out[1, 7], new[0]) and np.array_equal(out[1, 2], new[1])
    mask = np.ones(pool.shape[:2], bool)
    mask[1, 7] = mask[1, 2] = False
    assert np.array_equal(out[mask], pool[mask])


def pin_steady_predicate():
    assert R.is_steady_increment([4, 9], [10, 3], [4, 9], [11, 4])
    assert not R.is_steady_increment([4, 9], [10, 3], [9, 4], [4, 11])
    assert not R.is_steady_increment([4, 9], [10, 3], [4, 9], [11, 5])
    assert not R.is_steady_increment([4, 9], [10, 3], [4, 9, 2], [11, 4, 1])
    assert not R.is_steady_increment(None, None, [1], [1])


def pin_bf16_decode():
    # 1.0 = 0x3F80, -2.0 = 0xC000, 0.5 = 0x3F00, smallest subnormal 0x0001 = 2^-133.
    v = R.bf16_bits_to_f64(np.array([0x3F80, 0xC000, 0x3F00, 0x0001], dtype=np.uint16))
    assert list(v) == [1.0, -2.0, 0.5, 2.0 ** -133]


def pin_golden_extend():
    # Hand-worked causal means (tests/golden/extend_causal_means.json).
    g = _load("extend_causal_means.json")
    v0, v1 = g["V_request0"], g["V_request1"]
    V = np.array(v0 + v1, dtype=np.float64)[None, :, None, :]  # (1, slots, 1, 2)
    vb = _bits(V)
    kb = _bits(np.zeros_like(V))
    qb = _bits(np.array(g["q"], dtype=np.float64)[:, None, :])
    slots = [list(range(len(v0))), list(range(len(v0), len(v0) + len(v1)))]
    o, lse = R.extend_attention(qb, kb, vb, 0, slots, g["new_tokens"], g["scale"], 1)
    assert np.allclose(o[:, 0], _arr(g["o"]), rtol=0, atol=1e-13), o
    assert np.allclose(lse[:, 0], _arr(g["lse"]), rtol=0, atol=1e-13), lse


def _extend_case(seed=11, B=3, Hq=4, Hkv=2, D=8, P=4, lens=(6, 3, 9), qo=(2, 3, 4), NL=2):
    p = W.make_problem("tiny_extend", batch=B, n_layers=NL, n_q_heads=Hq, n_kv_heads=Hkv,
                       head_dim=D, page_size=P, seq_lens=list(lens), seed=seed)
    slots = [R.token_slots(b, int(p.seq_lens[b]), page_table=p.page_table.numpy(),
                           req_pool_indices=p.req_pool_indices.numpy(), page_size=P)
             for b in range(B)]
    q = W.normal_bf16((sum(qo), Hq, D), seed + 200)
    return p, slots, list(qo), q


def pin_extend_one_new_token_is_decode():
    # One new token per request: extend reduces to decode attention.
    p, q, slots, layer = _tiny_problem()
    kb, vb = R.tensor_bits(p.k_pool), R.tensor_bits(p.v_pool)
    od, ld = R.decode_attention(R.tensor_bits(q), kb, vb, layer, slots, p.scale, p.n_kv_heads)
    oe, le = R.extend_attention(R.tensor_bits(q), kb, vb, layer, slots, [1] * p.batch, p.scale,
                                p.n_kv_heads)
    assert np.array_equal(od, oe) and np.array_equal(ld, le)


def pin_extend_dense_causal():
    # Dense form: per request and head, S = Q K^T * scale with the positions
    # past each query masked, row softmax, times V, as whole matrices.
    p, slots, qo, q = _extend_case()
    layer = 1
    kb, vb = R.tensor_bits(p.k_pool), R.tensor_bits(p.v_pool)
    o, lse = R.extend_attention(R.tensor_bits(q), kb, vb, layer, slots, qo, p.scale,
                                p.n_kv_heads)
    qf = q.to(torch.float64).numpy()
    kf = p.k_pool.to(torch.float64).numpy()
    vf = p.v_pool.to(torch.float64).numpy()
    G = p.n_q_heads // p.n_kv_heads
    scale = float(np.float32(p.scale))
    r0 = 0
    for b, n in enumerate(qo):
        L = len(slots[b])
        sl = np.asarray(slots[b])
        for h in range(p.n_q_heads):
            K, V = kf[layer, sl, h // G], vf[layer, sl, h // G]
            Q = qf[r0:r0 + n, h]
            S = (Q @ K.T) * scale
            pos = np.arange(L - n, L)[:, None]
            S = np.where(np.arange(L)[None, :] > pos, -np.inf, S)
            Pm = np.exp(S - S.max(axis=1, keepdims=True))
            ref = (Pm @ V) / Pm.sum(axis=1, keepdims=True)
            assert np.allclose(o[r0:r0 + n, h], ref, rtol=0, atol=1e-12)
            ref_lse = S.max(axis=1) + np.log(Pm.sum(axis=1))
            assert np.allclose(lse[r0:r0 + n, h], ref_lse, rtol=0, atol=1e-12)
        r0 += n


def pin_extend_prefill_matches_sdpa():
    # Whole-context prefill (every token new) equals the float64 library
    # routine with its causal mask, K/V heads repeated for the groups.
    p, slots, _, _ = _extend_case(lens=(5, 8, 3))
    qo = [len(s) for s in slots]
    q = W.normal_bf16((sum(qo), p.n_q_heads, p.head_dim), 321)
    layer = 0
    o, _ = R.extend_attention(R.tensor_bits(q), R.tensor_bits(p.k_pool),
                              R.tensor_bits(p.v_pool), layer, slots, qo, p.scale,
                              p.n_kv_heads)
    G = p.n_q_heads // p.n_kv_heads
    r0 = 0
    for b, n in enumerate(qo):
        sl = torch.tensor(slots[b])
        K = p.k_pool[layer, sl].to(torch.float64).transpose(0, 1).repeat_interleave(G, 0)
        V = p.v_pool[layer, sl].to(torch.float64).transpose(0, 1).repeat_interleave(G, 0)
        Q = q[r0:r0 + n].to(torch.float64).transpose(0, 1)
        ref = torch.nn.functional.scaled_dot_product_attention(
            Q, K, V, is_causal=True, scale=float(np.float32(p.scale)))
        assert np.allclose(o[r0:r0 + n], ref.transpose(0, 1).numpy(), rtol=0, atol=1e-12)
        r0 += n


def pin_extend_causality():
    # A new token's output ignores rows after its position and depends on
    # the row at its position.
    p, slots, qo, q = _extend_case()
    layer = 1
    kb, vb = R.tensor_bits(p.k_pool).copy(), R.tensor_bits(p.v_pool).copy()
    qb = R.tensor_bits(q)
    o0, _ = R.extend_attention(qb, kb, vb, layer, slots, qo, p.scale, p.n_kv_heads)
    b = 2  # L = 9, new tokens at positions 5..8 -> query rows 5..8
    r_first = sum(qo[:b])
    k2, v2 = kb.copy(), vb.copy()
    # sign flips: the rows change and stay finite (an exponent-bit flip would
    # make Inf / NaN rows, which differ from anything)
    for t in range(6, 9):  # after the first new token's position (5)
        k2[layer, slots[b][t]] ^= np.uint16(0x8000)
        v2[layer, slots[b][t]] ^= np.uint16(0x8000)
    o1, _ = R.extend_attention(qb, k2, v2, layer, slots, qo, p.scale, p.n_kv_heads)
    assert np.array_equal(o0[r_first], o1[r_first])
    assert not np.allclose(o0[r_first + 1], o1[r_first + 1])
    k3 = kb.copy()
    k3[layer, slots[b][5]] ^= np.uint16(0x8000)
    o2, _ = R.extend_attention(qb, k3, vb, layer, slots, qo, p.scale, p.n_kv_heads)
    assert not np.allclose(o0[r_first], o2[r_first])


def pin_extend_append():
    p, slots, qo, _ = _extend_case()
    kb = R.tensor_bits(p.k_pool)
    new = np.arange(sum(qo) * p.n_kv_heads * p.head_dim, dtype=np.uint16).reshape(
        sum(qo), p.n_kv_heads, p.head_dim)
    out = R.extend_append(kb, 1, slots, qo, new)
    changed = {(1, int(s)) for b, n in enumerate(qo) for s in slots[b][len(slots[b]) - n:]}
    r = 0
    for b, n in enumerate(qo):
        for t in range(len(slots[b]) - n, len(slots[b])):
            assert np.array_equal(out[1, slots[b][t]], new[r])
            r += 1
    diff = np.argwhere(np.any(out != kb, axis=(2, 3)))
    assert {(int(a), int(c)) for a, c in diff} <= changed


def pin_token_slots_flat_golden():
    # Flat mode: token t of entry b is kv_indices[kv_indptr[b] + t], read here
    # from the hand-worked index of the flat bind fixture (not from bind).
    g = _load("bind_rebuild_flat.json")
    e = g["expect"]
    for b, want in enumerate(g["slots"]):
        got = R.token_slots(b, g["seq_lens"][b], index_mode=R.FLAT, kv_indptr=e["kv_indptr"],
                            kv_indices=e["kv_indices"])
        assert got == want, (b, got, want)


def pin_token_slots_flat_equals_table_walk():
    # With token-level pages (P = 1) the flat index built by the bind and the
    # request-to-token table walk name the same slots for every token.
    p = W.make_problem("flat", batch=4, n_layers=1, n_q_heads=2, n_kv_heads=1, head_dim=8,
                       page_size=1, seq_lens=[3, 1, 7, 5], seed=31)
    tbl, rows = p.page_table.numpy(), p.req_pool_indices.numpy()
    meta = R.bind(p.seq_lens.tolist(), req_pool_indices=rows, page_table=tbl, page_size=1,
                  mode=R.REBUILD, index_mode=R.FLAT)
    for b in range(p.batch):
        L = int(p.seq_lens[b])
        flat = R.token_slots(b, L, index_mode=R.FLAT, kv_indptr=meta["kv_indptr"],
                             kv_indices=meta["kv_indices"])
        walk = R.token_slots(b, L, page_table=tbl, req_pool_indices=rows, page_size=1)
        assert flat == walk, (b, flat, walk)


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


# ------------------------------------------------- planted mistakes -------

def _mut_gqa(h, n_q, n_kv):
    return h % n_kv


def _mut_attend_noscale(q, K, V, scale):
    return _orig["attend"](q, K, V, 1.0)


def _mut_attend_drop_last(q, K, V, scale):
    if K.shape[0] > 1:
        return _orig["attend"](q, K[:-1], V[:-1], scale)
    return _orig["attend"](q, K, V, scale)


def _mut_attend_sign(q, K, V, scale):
    return _orig["attend"](-q, K, V, scale)


def _mut_slot(b, t, *, page_table, req_pool_indices, page_size):
    row = int(req_pool_indices[b])
    return int(page_table[row][t // page_size]) + t % page_size


def _mut_merge_unweighted(ms, ls, os_):
    live = [s for s in range(len(ms)) if ls[s] > 0]
    if not live:
        return np.zeros(np.asarray(os_[0]).shape), -math.inf
    out = sum(np.asarray(os_[s]) * ls[s] for s in live) / sum(ls[s] for s in live)
    return out, max(ms[s] for s in live) + math.log(sum(ls[s] for s in live))


def _mut_token_slots_flat_next(b, seq_len, *, index_mode=R.PAGE_TABLE, kv_indptr=None,
                               kv_indices=None, **kw):
    if index_mode == R.FLAT:  # the next entry's base: kv_indptr[b + 1]
        base = int(kv_indptr[b + 1])
        return [int(kv_indices[(base + t) % len(kv_indices)]) for t in range(seq_len)]
    return _orig["token_slots"](b, seq_len, index_mode=index_mode, kv_indptr=kv_indptr,
                                kv_indices=kv_indices, **kw)


def _mut_bind_inclusive(seq_lens, **kw):
    res = _orig["bind"](seq_lens, **kw)
    res["kv_indptr"] = res["kv_indptr"][1:] + [res["kv_indptr"][-1]]
    return res


def _mut_bf16(bits):
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << np.uint32(15)
    return b.view(np.float32).astype(np.float64)


def _mut_positions_late(seq_len, n_new):
    return [min(seq_len - 1, seq_len - n_new + i + 1) for i in range(n_new)]


def _mut_positions_all(seq_len, n_new):
    return [seq_len - 1] * n_new


_orig = {"attend": R.attend, "bind": R.bind, "token_slots": R.token_slots}

MUTATIONS = {
    "gqa_modulo": ("kv_head_of", _mut_gqa),
    "scale_dropped": ("attend", _mut_attend_noscale),
    "new_token_not_attended": ("attend", _mut_attend_drop_last),
    "score_sign": ("attend", _mut_attend_sign),
    "slot_without_page_size": ("slot_of_token", _mut_slot),
    "merge_without_max_shift": ("merge", _mut_merge_unweighted),
    "indptr_inclusive": ("bind", _mut_bind_inclusive),
    "flat_slots_next_base": ("token_slots", _mut_token_slots_flat_next),
    "bf16_shift": ("bf16_bits_to_f64", _mut_bf16),
    "extend_position_shifted": ("extend_positions", _mut_positions_late),
    "extend_not_causal": ("extend_positions", _mut_positions_all),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistakes(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(R, attr, fn)
    caught = []
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"planted mistake {name} passed every pin"
