"""GPU parity of the paged extend (prefill) path: pkv_extend_append against
the oracle's append (bit-exact pool rows) and pkv_extend_attn against the
oracle's causal extend attention (max |err| <= 1e-2 and normwise <= 2e-2),
over page-table and flat indices, every group size the kernel has, ragged
new-token counts (0, 1, a partial query block, whole-context prefill), and
the device error paths.
"""
import numpy as np
import pytest
import torch

import oracle.ref as R
import pkv_inputs as W
from paged_kv_decode_bind_gb300 import CascadeDecoder, Workspace
from paged_kv_decode_bind_gb300 import _abi as A

from parity import check_attention

pytestmark = pytest.mark.gpu


def _slots(p):
    table, rows = p.page_table.numpy(), p.req_pool_indices.numpy()
    return [R.token_slots(b, int(p.seq_lens[b]), page_table=table, req_pool_indices=rows,
                          page_size=p.page_size) for b in range(p.batch)]


def _indptr(qo, device):
    return torch.tensor(np.concatenate([[0], np.cumsum(qo)]).astype(np.int32), device=device)


def run_extend(cuda, *, lens, qo, Hq, Hkv, D, P, seed, NL=2, layer=1, flags=0, rows=None,
               max_qo=None, table_edit=None, expect_err=0, check_pool=True, S=1):
    """Append + extend attention through libpkv and the oracle; returns the
    GPU output (float64 numpy) and the oracle's."""
    p = W.make_problem("extend", batch=len(lens), n_layers=NL, n_q_heads=Hq, n_kv_heads=Hkv,
                       head_dim=D, page_size=P, seq_lens=list(lens), seed=seed)
    if table_edit:
        table_edit(p)
    mq = max(qo) if max_qo is None else max_qo
    # split partials live in o_part / ml_part: room for batch * max_qo * S rows
    ws = Workspace.from_problem(p, max_splits=max(1, mq * S) if S > 1 else 1)
    B, T = p.batch, int(sum(qo))
    q = W.normal_bf16((T, Hq, D), seed + 500)
    kn = W.normal_bf16((T, Hkv, D), seed + 501)
    vn = W.normal_bf16((T, Hkv, D), seed + 502)
    if P == 1:
        A.pkv_bind_step(ws, B, A.PKV_BIND_REBUILD)  # kv_indptr and kv_indices
    qo_dev = _indptr(qo, cuda)
    out_dtype = torch.float32 if flags & A.PKV_FLAG_OUT_F32 else torch.bfloat16
    out = torch.full((T, Hq, D), 7.0, dtype=out_dtype, device=cuda)  # sentinel
    A.pkv_extend_append(ws, B, layer, qo_dev, mq, kn.to(cuda), vn.to(cuda))
    A.pkv_extend_attn(ws, B, layer, qo_dev, mq, q.to(cuda), out, p.scale, num_splits=S,
                      flags=flags)
    torch.cuda.synchronize()
    assert int(ws.err.item()) == expect_err
    slots = _slots(p)
    ok_req = [0 <= qo[b] <= lens[b] and qo[b] <= mq for b in range(B)]
    app_qo = [qo[b] if ok_req[b] else 0 for b in range(B)]
    # the oracle appends only for valid requests; rows of the others are skipped
    kb, vb = R.tensor_bits(p.k_pool), R.tensor_bits(p.v_pool)
    kb = R.extend_append(kb, layer, slots, app_qo, _rows_of(kn, qo, ok_req))
    vb = R.extend_append(vb, layer, slots, app_qo, _rows_of(vn, qo, ok_req))
    if check_pool:
        assert np.array_equal(R.tensor_bits(ws.k_pool.cpu()), kb), "K pool differs"
        assert np.array_equal(R.tensor_bits(ws.v_pool.cpu()), vb), "V pool differs"
    want = rows if rows is not None else [(r, h) for r in range(T) for h in range(Hq)]
    ref, _ = R.extend_attention(R.tensor_bits(q), kb, vb, layer, slots, qo, p.scale, Hkv,
                                rows=want)
    got = out.to(torch.float64).cpu().numpy()
    return got, ref, want, p


def _rows_of(x, qo, ok_req):
    """The new-token rows of the valid requests, in request order (bits)."""
    bits = R.tensor_bits(x)
    keep, r = [], 0
    for b, n in enumerate(qo):
        if ok_req[b]:
            keep.extend(range(r, r + n))
        r += n
    return bits[keep] if keep else bits[:0]


def _compare(got, ref, want, what):
    g = np.stack([got[r, h] for r, h in want])
    e = np.stack([ref[r, h] for r, h in want])
    return check_attention(g, e, what)


CASES = {
    # name: (lens, qo, Hq, Hkv, D, P)
    "paged_g4_d128": ((70, 200, 33), (5, 64, 33), 32, 8, 128, 16),
    "paged_g1_d64_zero_and_one": ((90, 17, 40), (17, 1, 0), 4, 4, 64, 16),
    "flat_g8_d128": ((150, 90, 1), (20, 9, 1), 16, 2, 128, 1),
    "paged8_g16_d128": ((61, 100), (3, 5), 32, 2, 128, 8),
    "prefill_g2_d64": ((37, 130), (37, 130), 8, 4, 64, 16),
    "paged_g8_d64_partial_block": ((300, 129), (13, 129), 16, 2, 64, 16),
}


# the kernel pkv_extend_attn picks (tcgen05 where page sizes are a multiple
# of 16, else the warp-level one), and the warp-level one by request
KERNS = {"auto": 0, "warp": A.PKV_FLAG_EXTEND_WARP_MMA}


@pytest.mark.parametrize("kern", list(KERNS))
@pytest.mark.parametrize("S", [1, 3])
@pytest.mark.parametrize("case", list(CASES), ids=list(CASES))
def test_extend_parity(cuda, case, S, kern):
    lens, qo, Hq, Hkv, D, P = CASES[case]
    got, ref, want, _ = run_extend(cuda, lens=lens, qo=qo, Hq=Hq, Hkv=Hkv, D=D, P=P, seed=4100,
                                   S=S, flags=KERNS[kern])
    _compare(got, ref, want, f"{case} S={S} {kern}")


@pytest.mark.parametrize("kern,bar", [("auto", 1e-3), ("warp", 2e-3)])
def test_extend_splits_agree(cuda, kern, bar):
    # fp32 outputs of 1, 2, 5 and 16 splits (some of them empty for early
    # query blocks) agree with each other.  The tcgen05 kernel applies P as
    # bf16 high and low parts (~2^-17 of each weight): 1e-3.  The warp-level
    # kernel rounds P to one bf16, which depends on the running maximum: 2e-3.
    kw = dict(lens=(1500, 700), qo=(48, 100), Hq=16, Hkv=2, D=128, P=16, seed=4700, NL=1,
              layer=0, flags=A.PKV_FLAG_OUT_F32 | KERNS[kern],
              rows=[(r, h) for r in range(0, 148, 7) for h in range(16)])
    outs = []
    for S in (1, 2, 5, 16):
        got, ref, want, _ = run_extend(cuda, S=S, **kw)
        _compare(got, ref, want, f"S={S}")
        outs.append(got)
    for o in outs[1:]:
        assert np.abs(o - outs[0]).max() <= bar


def test_extend_kernels_agree(cuda):
    # fp32 outputs of the tcgen05 and the warp-level kernel, same inputs.  The
    # tcgen05 kernel's P = P_hi + P_lo keeps it within 1e-3 of the fp64
    # oracle; the warp-level kernel's single bf16 P moves it by up to a few
    # 1e-3, so the two agree within 5e-3.
    kw = dict(lens=(900, 333, 64), qo=(200, 33, 64), Hq=32, Hkv=8, D=128, P=16, seed=5000,
              NL=1, layer=0)
    a, ref, _, _ = run_extend(cuda, flags=A.PKV_FLAG_OUT_F32, **kw)
    b, _, _, _ = run_extend(cuda, flags=A.PKV_FLAG_OUT_F32 | A.PKV_FLAG_EXTEND_WARP_MMA, **kw)
    assert np.abs(a - ref).max() <= 1e-3
    assert np.abs(a - b).max() <= 5e-3


def test_extend_many_units_per_cta(cuda):
    # More (query block, request, KV head) units than CTAs: every CTA runs
    # several units back to back through the same barriers and tensor memory.
    lens, qo = (700, 420, 900, 512, 300, 640), (256, 256, 200, 256, 256, 100)
    rng = np.random.default_rng(5)
    T = sum(qo)
    rows = sorted({(int(rng.integers(T)), int(rng.integers(32))) for _ in range(300)}
                  | {(0, 0), (T - 1, 31)})
    for S in (1, 2):
        got, ref, want, _ = run_extend(cuda, lens=lens, qo=qo, Hq=32, Hkv=8, D=128, P=16,
                                       seed=5100, NL=1, layer=0, rows=rows, S=S)
        _compare(got, ref, want, f"many units S={S}")


def test_extend_running_max_jumps(cuda):
    # Key rows scaled x40 part-way through each context lift the scores by
    # far more than 2^8: the tcgen05 kernel raises its reference maximum and
    # rescales O in tensor memory.  Outputs against the oracle, both kernels.
    def edit(p):
        table, rows = p.page_table, p.req_pool_indices
        for b in range(p.batch):
            L = int(p.seq_lens[b])
            for t in (L // 3, L // 2 + 5, L - 70):
                page = int(table[int(rows[b]), t // p.page_size])
                slot = page * p.page_size + t % p.page_size
                p.k_pool[:, slot] = (p.k_pool[:, slot].float() * 40).to(torch.bfloat16)
    for kern in KERNS.values():
        got, ref, want, _ = run_extend(cuda, lens=(600, 1000), qo=(100, 300), Hq=16, Hkv=2,
                                       D=128, P=16, seed=5200, NL=1, layer=0, table_edit=edit,
                                       flags=A.PKV_FLAG_OUT_F32 | kern)
        _compare(got, ref, want, f"outlier keys {kern}")


def test_extend_f32_output_one_new_token(cuda):
    # One new token per request with fp32 output; the bf16 output is its
    # round-to-nearest-even.
    lens, qo = (45, 130, 8), (1, 1, 1)
    got, ref, want, p = run_extend(cuda, lens=lens, qo=qo, Hq=32, Hkv=8, D=128, P=16, seed=4200,
                                   flags=A.PKV_FLAG_OUT_F32)
    _compare(got, ref, want, "f32")
    gb, _, _, _ = run_extend(cuda, lens=lens, qo=qo, Hq=32, Hkv=8, D=128, P=16, seed=4200)
    rb = torch.tensor(got).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(gb, rb)


def test_extend_long_prefix_sampled(cuda):
    # A 4096-token prefix with a 256-token chunk: many tiles per unit,
    # compared on sampled rows.  40 splits: rows of more than 32 partials,
    # merged in two chunks, and (the 700-token request's splits past its
    # end) units without tiles between units with tiles in a CTA's list.
    rng = np.random.default_rng(3)
    T = 256 + 64
    rows = sorted({(int(rng.integers(T)), int(rng.integers(32))) for _ in range(40)}
                  | {(0, 0), (T - 1, 31), (255, 5)})
    for S in (1, 6, 40):
        got, ref, want, _ = run_extend(cuda, lens=(4096, 700), qo=(256, 64), Hq=32, Hkv=8,
                                       D=128, P=16, seed=4300, NL=1, layer=0, rows=rows, S=S)
        _compare(got, ref, want, f"long prefix S={S}")


def test_extend_invalid_request_is_skipped(cuda):
    # Request 0 claims more new tokens than it holds: PKV_DEVERR_LEN, its rows
    # keep the sentinel and nothing of it is appended; request 1 is exact.
    lens, qo = (10, 40), (12, 6)
    got, ref, want, _ = run_extend(cuda, lens=lens, qo=qo, Hq=8, Hkv=2, D=64, P=16, seed=4400,
                                   expect_err=A.PKV_DEVERR_LEN,
                                   rows=[(r, h) for r in range(12, 18) for h in range(8)])
    assert np.all(got[:12] == 7.0)
    _compare(got, ref, want, "valid request next to an invalid one")


def test_extend_max_qo_len_too_small(cuda):
    lens, qo = (50, 40), (9, 3)
    got, ref, want, _ = run_extend(cuda, lens=lens, qo=qo, Hq=8, Hkv=2, D=64, P=16, seed=4500,
                                   max_qo=4, expect_err=A.PKV_DEVERR_LEN,
                                   rows=[(r, h) for r in range(9, 12) for h in range(8)])
    assert np.all(got[:9] == 7.0)
    _compare(got, ref, want, "request within max_qo_len")


def test_extend_bad_page_zeroes_rows(cuda):
    # Request 1's first page id is out of range: PKV_DEVERR_PAGE and its rows
    # are zeros (every unit of it reads page 0); request 0 stays exact.
    def edit(p):
        row = int(p.req_pool_indices[1])
        p.page_table[row, 0] = p.pool_slots // p.page_size  # one past the last page
    lens, qo = (64, 80), (8, 8)
    for S in (1, 2):
        got, ref, want, _ = run_extend(cuda, lens=lens, qo=qo, Hq=8, Hkv=2, D=64, P=16,
                                       seed=4600, table_edit=edit, expect_err=A.PKV_DEVERR_PAGE,
                                       check_pool=False, S=S,
                                       rows=[(r, h) for r in range(8) for h in range(8)])
        assert np.all(got[8:] == 0.0)
        _compare(got, ref, want, f"request next to a bad page S={S}")


def test_extend_graph_replay_bitexact(cuda):
    # The extend calls allocate nothing and read no device memory on the
    # host: a captured graph replays them with bit-identical outputs.
    p = W.make_problem("extend_graph", batch=2, n_layers=1, n_q_heads=16, n_kv_heads=2,
                       head_dim=128, page_size=16, seq_lens=[300, 130], seed=4800)
    qo = [40, 130]
    S = 3
    ws = Workspace.from_problem(p, max_splits=max(qo) * S)
    T = sum(qo)
    q = W.normal_bf16((T, 16, 128), 4801).to(cuda)
    kn = W.normal_bf16((T, 2, 128), 4802).to(cuda)
    vn = W.normal_bf16((T, 2, 128), 4803).to(cuda)
    qo_dev = _indptr(qo, cuda)
    out = torch.zeros((T, 16, 128), dtype=torch.bfloat16, device=cuda)

    def step(s=None):
        A.pkv_extend_append(ws, 2, 0, qo_dev, max(qo), kn, vn, stream=s)
        A.pkv_extend_attn(ws, 2, 0, qo_dev, max(qo), q, out, p.scale, num_splits=S, stream=s)

    step()
    torch.cuda.synchronize()
    eager = out.clone()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side), torch.cuda.graph(g, stream=side):
        step(side)
    torch.cuda.current_stream().wait_stream(side)
    g.replay()
    torch.cuda.synchronize()
    assert int(ws.err.item()) == 0
    assert torch.equal(out, eager)


@pytest.mark.parametrize("S,full,big", [(1, False, False), (2, False, False), (1, True, False),
                                        (3, False, True)])
def test_extend_plan_early_layers(cuda, S, full, big):
    # Layers after the first with PKV_FLAG_PLAN_EARLY: with CTA slots to
    # spare the tcgen05 kernel orders its units and loads the cached tokens'
    # K/V before the previous launch (this layer's append) ends; a grid that
    # fills every slot launches plainly and ignores the flag.  Outputs equal
    # those of plain launches bit for bit, eagerly and replayed from a graph.
    NL, lens, qo = 3, [900, 1500, 700, 1200], [64, 40, 64, 17]
    if full:
        lens, qo = [1500, 900, 700, 1200], [32, 32, 32, 32]
    if big:  # 672 units: several per CTA
        qo = [200, 96, 160, 64]
    p = W.make_problem("extend_early", batch=4, n_layers=NL, n_q_heads=32, n_kv_heads=8,
                       head_dim=128, page_size=16, seq_lens=lens, seed=6100 + S)
    T, mq = sum(qo), max(qo)
    q = [W.normal_bf16((T, 32, 128), 6200 + l).to(cuda) for l in range(NL)]
    kn = [W.normal_bf16((T, 8, 128), 6300 + l).to(cuda) for l in range(NL)]
    vn = [W.normal_bf16((T, 8, 128), 6400 + l).to(cuda) for l in range(NL)]
    qo_dev = _indptr(qo, cuda)
    base = A.PKV_FLAG_EXTEND_FULL if full else 0

    def run(early, graph):
        ws = Workspace.from_problem(p, max_splits=mq * S if S > 1 else 1)
        out = torch.zeros((NL, T, 32, 128), dtype=torch.bfloat16, device=cuda)

        def step(s=None):
            for l in range(NL):
                if not full:  # the cascade's prefix pass has no new tokens in the pool
                    A.pkv_extend_append(ws, 4, l, qo_dev, mq, kn[l], vn[l], stream=s)
                fl = base | (A.PKV_FLAG_PLAN_EARLY if early and l > 0 else 0)
                A.pkv_extend_attn(ws, 4, l, qo_dev, mq, q[l], out[l], p.scale, num_splits=S,
                                  flags=fl, stream=s)

        if graph:
            g = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side), torch.cuda.graph(g, stream=side):
                step(side)
            torch.cuda.current_stream().wait_stream(side)
            for _ in range(2):
                g.replay()
        else:
            step()
        torch.cuda.synchronize()
        assert int(ws.err.item()) == 0
        return out

    ref = run(False, False)
    assert torch.equal(run(True, False), ref)
    assert torch.equal(run(True, True), ref)
    # the plain launches against the oracle on a sample of layer 2's rows
    slots = _slots(p)
    kb, vb = R.tensor_bits(p.k_pool), R.tensor_bits(p.v_pool)
    rng = np.random.default_rng(6500 + S + 2 * big)
    rows = sorted({(int(rng.integers(T)), int(rng.integers(32))) for _ in range(40)})
    if full:
        qb = R.tensor_bits(q[2].cpu())
        r0, parts = 0, []
        for b in range(4):
            o, _ = R.decode_attention(qb[r0:r0 + qo[b]], kb, vb, 2, [slots[b][:lens[b]]] * qo[b],
                                      p.scale, 8)
            parts.append(o)
            r0 += qo[b]
        _compare(ref[2].to(torch.float64).cpu().numpy(), np.concatenate(parts), rows,
                 "early full")
    else:
        kb = R.extend_append(kb, 2, slots, qo, R.tensor_bits(kn[2].cpu()))
        vb = R.extend_append(vb, 2, slots, qo, R.tensor_bits(vn[2].cpu()))
        oracle_out, _ = R.extend_attention(R.tensor_bits(q[2].cpu()), kb, vb, 2, slots, qo,
                                           p.scale, 8, rows=rows)
        _compare(ref[2].to(torch.float64).cpu().numpy(), oracle_out, rows, f"early S={S}")


def test_extend_one_token_matches_decode_kernel(cuda):
    # One new token per request: the extend kernel and the decode kernel
    # compute the same attention; their fp32 outputs agree to the extend
    # kernel's bf16 rounding of P.
    lens = [700, 65, 1200]
    p = W.make_problem("extend_vs_decode", batch=3, n_layers=1, n_q_heads=32, n_kv_heads=8,
                       head_dim=128, page_size=16, seq_lens=lens, seed=4900)
    ws = Workspace.from_problem(p)
    q = W.normal_bf16((3, 32, 128), 4901).to(cuda)
    qo_dev = _indptr([1, 1, 1], cuda)
    out = torch.zeros((3, 32, 128), dtype=torch.float32, device=cuda)
    A.pkv_extend_attn(ws, 3, 0, qo_dev, 1, q, out, p.scale, flags=A.PKV_FLAG_OUT_F32)
    A.pkv_decode_attn(ws, 3, 0, q, p.scale, 1, A.PKV_FLAG_OUT_F32)
    torch.cuda.synchronize()
    assert int(ws.err.item()) == 0
    dec = ws.out_f32(3)
    assert (out - dec).abs().max().item() <= 2e-3


@pytest.mark.parametrize("Sp,Ss", [(1, 1), (4, 2)])
def test_cascade_shared_prefix(cuda, Sp, Ss):
    # Requests whose first 512 tokens alias the same pages: the cascade
    # (shared prefix once + own suffix + merge) equals decode attention over
    # each request's whole context.
    B, prefix_len = 8, 512
    lens = [prefix_len + x for x in (40, 1, 130, 77, 200, 16, 95, 3)]
    p = W.make_problem("cascade", batch=B, n_layers=2, n_q_heads=32, n_kv_heads=8,
                       head_dim=128, page_size=16, seq_lens=lens, seed=5100)
    rows = p.req_pool_indices.tolist()
    shared = p.page_table[rows[0], :prefix_len // 16].clone()
    for b in range(1, B):
        p.page_table[rows[b], :prefix_len // 16] = shared
    ws = Workspace.from_problem(p, max_splits=max(2, Ss))
    q = W.normal_bf16((B, 32, 128), 5101)
    cas = CascadeDecoder(ws, B, prefix_len, scale=p.scale, prefix_splits=Sp, suffix_splits=Ss)
    out = torch.zeros((B, 32, 128), dtype=torch.float32, device=cuda)
    # the suffix attention on a second stream when the prefix is split
    cas.layer(1, q.to(cuda), out, flags=A.PKV_FLAG_OUT_F32,
              suffix_stream=torch.cuda.Stream() if Sp > 1 else None)
    torch.cuda.synchronize()
    assert int(ws.err.item()) == 0
    ref, _ = R.decode_attention(R.tensor_bits(q), R.tensor_bits(p.k_pool), R.tensor_bits(p.v_pool),
                                1, _slots(p), p.scale, 8)
    check_attention(out.to(torch.float64).cpu().numpy(), ref, f"cascade Sp={Sp} Ss={Ss}")


def test_cascade_steady_step(cuda):
    # A steady decode step through the cascade: its bind advances the suffix
    # lengths and appends the new rows past the prefix; the attention then
    # equals decode over the whole grown contexts.
    B, prefix_len = 6, 256
    lens = [prefix_len + x for x in (30, 1, 100, 64, 7, 150)]
    p = W.make_problem("cascade_step", batch=B, n_layers=2, n_q_heads=16, n_kv_heads=2,
                       head_dim=128, page_size=16, seq_lens=lens, steps=1, seed=5200)
    rows = p.req_pool_indices.tolist()
    shared = p.page_table[rows[0], :prefix_len // 16].clone()
    for b in range(1, B):
        p.page_table[rows[b], :prefix_len // 16] = shared
    ws = Workspace.from_problem(p, max_splits=2)
    q, k, v = W.step_inputs(p, 0)
    cas = CascadeDecoder(ws, B, prefix_len, scale=p.scale, prefix_splits=2)
    cas.bind(A.PKV_BIND_STEADY, 0, 2, k.to(cuda), v.to(cuda))
    out = torch.zeros((B, 16, 128), dtype=torch.bfloat16, device=cuda)
    cas.layer(1, q[1].to(cuda), out)
    torch.cuda.synchronize()
    assert int(ws.err.item()) == 0
    assert cas.suffix_lens.tolist() == [x - prefix_len + 1 for x in lens]
    meta = R.bind(lens, req_pool_indices=p.req_pool_indices.numpy(),
                  page_table=p.page_table.numpy(), page_size=16, mode=R.STEADY)
    kb, vb = R.tensor_bits(p.k_pool), R.tensor_bits(p.v_pool)
    for layer in range(2):
        kb = R.append_rows(kb, layer, meta["out_loc"], R.tensor_bits(k)[layer])
        vb = R.append_rows(vb, layer, meta["out_loc"], R.tensor_bits(v)[layer])
    assert np.array_equal(R.tensor_bits(ws.k_pool.cpu()), kb)
    slots = [R.token_slots(b, meta["seq_lens"][b], page_table=p.page_table.numpy(),
                           req_pool_indices=p.req_pool_indices.numpy(), page_size=16)
             for b in range(B)]
    ref, _ = R.decode_attention(R.tensor_bits(q)[1], kb, vb, 1, slots, p.scale, 2)
    check_attention(out.to(torch.float64).cpu().numpy(), ref, "cascade steady step")


def test_cascade_graph_branch_bitexact(cuda):
    # The cascade captured in a CUDA graph with its suffix attention on a
    # parallel branch replays to the eager result bit for bit.
    B, prefix_len = 8, 256
    lens = [prefix_len + x for x in (9, 70, 33, 1, 120, 64, 5, 200)]
    p = W.make_problem("cascade_graph", batch=B, n_layers=1, n_q_heads=32, n_kv_heads=8,
                       head_dim=128, page_size=16, seq_lens=lens, seed=5300,
                       shared_prefix_pages=prefix_len // 16)
    ws = Workspace.from_problem(p, max_splits=2)
    q = W.normal_bf16((B, 32, 128), 5301).to(cuda)
    cas = CascadeDecoder(ws, B, prefix_len, scale=p.scale, prefix_splits=4)
    out = torch.zeros((B, 32, 128), dtype=torch.bfloat16, device=cuda)
    branch = torch.cuda.Stream()
    cas.layer(0, q, out, suffix_stream=branch)
    torch.cuda.synchronize()
    eager = out.clone()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side), torch.cuda.graph(g, stream=side):
        cas.layer(0, q, out, stream=side, suffix_stream=branch)
    torch.cuda.current_stream().wait_stream(side)
    g.replay()
    torch.cuda.synchronize()
    assert int(ws.err.item()) == 0
    assert torch.equal(out, eager)
    ref, _ = R.decode_attention(R.tensor_bits(q.cpu()), R.tensor_bits(p.k_pool),
                                R.tensor_bits(p.v_pool), 0, _slots(p), p.scale, 8)
    check_attention(out.to(torch.float64).cpu().numpy(), ref, "cascade graph")


def test_extend_full_mode_more_rows_than_keys(cuda):
    # Full mode: 40 query rows over a 16-token context (rows are not context
    # tokens), and an empty context (zero rows, lse -inf), without error bits.
    p = W.make_problem("full", batch=2, n_layers=1, n_q_heads=8, n_kv_heads=2, head_dim=64,
                       page_size=16, seq_lens=[16, 32], seed=5400)
    ws = Workspace.from_problem(p)
    ws.seq_lens[1] = 0  # request 1: no context at all
    qo = [40, 3]
    T = sum(qo)
    lse = torch.zeros(T * 8, dtype=torch.float32, device=cuda)
    view = A.PkvWorkspace.from_buffer_copy(ws.struct)
    view.lse, view.max_batch = lse.data_ptr(), 2 * max(qo)
    q = W.normal_bf16((T, 8, 64), 5401)
    out = torch.full((T, 8, 64), 7.0, dtype=torch.float32, device=cuda)
    A.pkv_extend_attn(view, 2, 0, _indptr(qo, cuda), max(qo), q.to(cuda), out, p.scale,
                      flags=A.PKV_FLAG_EXTEND_FULL | A.PKV_FLAG_OUT_F32 | A.PKV_FLAG_WRITE_LSE)
    torch.cuda.synchronize()
    assert int(ws.err.item()) == 0
    slots = _slots(p)
    qb = R.tensor_bits(q)
    kb, vb = R.tensor_bits(p.k_pool), R.tensor_bits(p.v_pool)
    # every row of request 0 attends its whole 16-token context: decode
    # attention of each row as its own one-token query
    ref, ref_lse = R.decode_attention(qb[:40], kb, vb, 0, [slots[0]] * 40, p.scale, 2)
    got = out.to(torch.float64).cpu().numpy()
    check_attention(got[:40], ref, "full mode")
    lse_got = lse.cpu().numpy().reshape(T, 8)
    assert np.abs(lse_got[:40] - ref_lse).max() < 1e-3
    assert np.all(got[40:] == 0.0)
    assert np.all(np.isneginf(lse_got[40:]))


def test_extend_rows_past_workspace_rejected(cuda):
    # With splits the partials live in the workspace, sized for batch *
    # max_qo_len new tokens.  Request 0 (9 tokens, max_qo_len 4) is invalid and
    # pushes request 1's rows to 9..11, past the 8 rows held: request 1 is
    # rejected too, and neither request's rows are written.
    got, _, _, _ = run_extend(cuda, lens=(50, 40), qo=(9, 3), Hq=8, Hkv=2, D=64, P=16,
                              seed=4500, max_qo=4, expect_err=A.PKV_DEVERR_LEN, rows=[], S=3)
    assert np.all(got == 7.0)


def _merge_lse_inputs(n, D, seed):
    """Two parts' outputs and lse over n rows: finite on both sides, one side
    empty (-inf), both empty, equal lse, and one side larger by 40."""
    rng = np.random.default_rng(seed)
    oa = rng.standard_normal((n, D)).astype(np.float32)
    ob = rng.standard_normal((n, D)).astype(np.float32)
    la = rng.uniform(-6.0, 6.0, n).astype(np.float32)
    lb = rng.uniform(-6.0, 6.0, n).astype(np.float32)
    la[3] = -np.inf
    lb[5] = -np.inf
    la[7] = lb[7] = -np.inf
    la[11] = lb[11] = 2.5
    lb[13] = la[13] + 40.0
    return oa, la, ob, lb


def _merge_lse_check(oa, la, ob, lb, got, got_lse, out_f32):
    """Compare with the oracle's log-sum-exp merge of the two parts (each
    part's lse as its max, with a unit sum; an empty part has sum 0)."""
    n, D = oa.shape
    ref, ref_lse = np.zeros((n, D)), np.zeros(n)
    for r in range(n):
        ms = [float(la[r]), float(lb[r])]
        ls = [0.0 if np.isneginf(m) else 1.0 for m in ms]
        ref[r], ref_lse[r] = R.merge(ms, ls, [oa[r].astype(np.float64), ob[r].astype(np.float64)])
    # fp32 arithmetic on O(1) values; bf16 output adds its rounding (2^-9 relative)
    tol = 2e-5 + (0.0 if out_f32 else 2.0 ** -8) * np.abs(ref)
    assert np.all(np.abs(got - ref) <= tol), float(np.abs(got - ref).max())
    both_empty = np.isneginf(la) & np.isneginf(lb)
    assert np.all(np.isneginf(got_lse[both_empty])) and np.all(got[both_empty] == 0.0)
    fin = ~both_empty
    assert np.all(np.abs(got_lse[fin] - ref_lse[fin]) <= 2e-5)


@pytest.mark.parametrize("D,out_f32", [(64, True), (128, False), (256, True)])
def test_merge_lse_two_way(cuda, D, out_f32):
    # 37 rows: a ragged last block of four rows
    oa, la, ob, lb = _merge_lse_inputs(37, D, 5500 + D)
    dt = torch.float32 if out_f32 else torch.bfloat16
    out = torch.full(oa.shape, 7.0, dtype=dt, device=cuda)
    lse = torch.full((oa.shape[0],), 7.0, dtype=torch.float32, device=cuda)
    dev = [torch.from_numpy(x).to(cuda) for x in (oa, la, ob, lb)]
    A.pkv_merge_lse(oa.shape[0], D, dev[0], dev[1], dev[2], dev[3], out, lse,
                    A.PKV_FLAG_OUT_F32 if out_f32 else 0)
    torch.cuda.synchronize()
    _merge_lse_check(oa, la, ob, lb, out.to(torch.float64).cpu().numpy(),
                     lse.to(torch.float64).cpu().numpy(), out_f32)


def test_cascade_suffix_past_its_row_is_rejected(cuda):
    # The suffix view's table rows start past the prefix's pages, so a
    # suffix may hold only the rest of a row.  Request 1 fills its whole row
    # (16 pages); the steady bind's +1 takes its suffix past the 12 pages left
    # after the 4-page prefix: the bind raises PKV_DEVERR_LEN and gives it no
    # slot, instead of reading the next row's first page id.
    B, prefix_len = 3, 64
    lens = [prefix_len + 40, 16 * 16, prefix_len + 100]
    p = W.make_problem("cascade_cap", batch=B, n_layers=1, n_q_heads=8, n_kv_heads=2,
                       head_dim=128, page_size=16, seq_lens=lens, seed=5400,
                       shared_prefix_pages=prefix_len // 16)
    assert p.max_pages_per_req == 16
    ws = Workspace.from_problem(p)
    cas = CascadeDecoder(ws, B, prefix_len, scale=p.scale)
    assert cas.suffix_view.max_seq_len == 12 * 16
    cas.bind(A.PKV_BIND_STEADY)
    torch.cuda.synchronize()
    assert int(ws.err.item()) & A.PKV_DEVERR_LEN
    assert cas.suffix_out_loc[1].item() == -1
    # the other two requests' slots, from the oracle over the suffix table
    meta = R.bind([lens[0] - prefix_len, lens[2] - prefix_len],
                  req_pool_indices=p.req_pool_indices.numpy()[[0, 2]],
                  page_table=p.page_table[:, prefix_len // 16:].contiguous().numpy(),
                  page_size=16, mode=R.STEADY)
    got = cas.suffix_out_loc.tolist()
    assert [got[0], got[2]] == meta["out_loc"]
