"""GPU parity: libpkv against the CPU fp64 oracle on the same seeded inputs.

Small cases (oracle-sized variants of every workload, several tiles and a
ragged tail) compare every output element; full-size cases run the launch
configuration the benchmark uses and compare metadata fully and attention on
sampled (request, head) pairs.
"""
import numpy as np
import pytest
import torch

import oracle.ref as R
import pkv_inputs as W
from paged_kv_decode_bind_gb300 import BindTracker, DecodeRunner, Workspace
from paged_kv_decode_bind_gb300 import _abi as A

from parity import OracleState, bf16_to_f64, check_attention, check_meta, run_steps

pytestmark = pytest.mark.gpu

SIMT, MMA, GATHER = A.PKV_FLAG_FORCE_SIMT, A.PKV_FLAG_FORCE_MMA, A.PKV_FLAG_FORCE_GATHER
FIXED = A.PKV_FLAG_FIXED_CHUNK
# (flags, fused): the CUDA-core kernel; the tensor-core kernel with TMA boxes
# (page sizes that are multiples of 16) or cp.async gathers; the fused layer
# kernel (append + attention + merge in one launch) with either producer and
# apportioned splits, and with the fixed chunks of the unfused call.
PATHS = {"simt": (SIMT, False), "mma": (MMA, False), "gather": (MMA | GATHER, False),
         "fused": (0, True), "fused_gather": (GATHER, True), "fused_fixed": (FIXED, True)}
KERNELS = pytest.mark.parametrize("kern", list(PATHS), ids=list(PATHS))


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _sample_heads(p, n, seed=0):
    rng = np.random.default_rng(seed)
    pairs = {(int(rng.integers(p.batch)), int(rng.integers(p.n_q_heads))) for _ in range(n)}
    pairs |= {(p.batch - 1, p.n_q_heads - 1), (0, 0)}
    return sorted(pairs)


# ---------------------------------------------------------------- small ----

def test_single_d64_full(cuda):
    # The whole single-request D=64 workload is oracle-sized: every element.
    p = W.workload("single_d64", steps=1)
    r = run_steps(p, S=1, check_pool=True)
    assert r["max_err"] <= 1e-2


@KERNELS
@pytest.mark.parametrize("S", [1, 3, 8])
def test_paged_gqa4_small(cuda, S, kern):
    p = W.workload("gqa4_b4_paged", shrink=8, steps=1)
    run_steps(p, S=S, check_partials=True, check_pool=True, flags=PATHS[kern][0],
                  fused=PATHS[kern][1])


@KERNELS
@pytest.mark.parametrize("S", [1, 5])
def test_flat_skewed_small(cuda, S, kern):
    p = W.workload("gqa4_b16_flat_skewed", shrink=16, steps=1)
    run_steps(p, S=S, check_partials=True, check_pool=True, flags=PATHS[kern][0],
                  fused=PATHS[kern][1])


@KERNELS
@pytest.mark.parametrize("B,S", [(1, 16), (4, 7)])
def test_long_small(cuda, B, S, kern):
    p = W.workload("gqa4_long_65536", batch=B, shrink=64, steps=1)
    run_steps(p, S=S, check_partials=True, flags=PATHS[kern][0], fused=PATHS[kern][1])


@KERNELS
@pytest.mark.parametrize("B,S", [(1, 1), (4, 4), (16, 2)])
def test_gqa8_small(cuda, B, S, kern):
    p = W.workload("gqa8_graph_sweep", batch=B, shrink=16, steps=1)
    run_steps(p, S=S, check_partials=True, check_pool=True, flags=PATHS[kern][0],
                  fused=PATHS[kern][1])


@KERNELS
@pytest.mark.parametrize("G,D", [(1, 128), (2, 64), (8, 64), (4, 64), (16, 128), (16, 64)])
def test_group_and_head_dim_variants(cuda, G, D, kern):
    if G == 16 and kern == "simt":
        pytest.skip("the CUDA-core kernel covers G <= 8")
    Hkv = 2
    p = W.make_problem("variant", batch=3, n_layers=2, n_q_heads=G * Hkv, n_kv_heads=Hkv,
                       head_dim=D, page_size=16, seq_lens=[1, 77, 200], seed=99, steps=1)
    for S in (1, 4):
        run_steps(p, S=S, check_partials=True, check_pool=True, flags=PATHS[kern][0],
                  fused=PATHS[kern][1])


@KERNELS
@pytest.mark.parametrize("P", [1, 4, 32])
def test_page_sizes(cuda, P, kern):
    p = W.make_problem("pages", batch=4, n_layers=1, n_q_heads=8, n_kv_heads=2, head_dim=128,
                       page_size=P, seq_lens=[33, 1, 130, 64], seed=123 + P,
                       index_mode=W.INDEX_PAGE_TABLE, steps=1)
    for S in (1, 3):
        run_steps(p, S=S, check_partials=True, check_pool=True, flags=PATHS[kern][0],
                  fused=PATHS[kern][1])


@pytest.mark.parametrize("fused", [False, True])
def test_multi_step_steady(cuda, fused):
    # 64 consecutive steady steps (+1 token each); the last step is compared.
    p = W.workload("gqa4_b4_paged", shrink=16, n_layers=1, steps=64)
    r = run_steps(p, S=4, steps=64, check_pool=True, fused=fused)
    ws = r["ws"]
    assert ws.seq_lens[:p.batch].tolist() == [x + 64 for x in p.seq_lens.tolist()]


def test_cross_split_agreement(cuda):
    # fp32 outputs from different split counts agree within 1e-3.
    p = W.workload("gqa4_long_65536", batch=2, shrink=32, steps=1)
    outs = []
    # (64 splits: rows of more than 32 partials, merged in two chunks)
    for S, fused, fl in ((1, False, 0), (2, False, 0), (9, False, 0), (32, False, 0),
                         (64, False, 0), (2, True, 0), (9, True, 0), (32, True, 0),
                         (64, True, 0), (9, True, FIXED)):
        ws = Workspace.from_problem(p, max_splits=S)
        run = DecodeRunner(ws, p.batch, num_splits=S, flags=A.PKV_FLAG_OUT_F32 | fl,
                           scale=p.scale, fused=fused)
        q, k, v = W.step_inputs(p, 0)
        run.q_in.copy_(q), run.k_in.copy_(k), run.v_in.copy_(v)
        run.step()
        torch.cuda.synchronize()
        outs.append(ws.out_f32(p.batch).cpu().numpy())
    for o in outs[1:]:
        assert np.abs(o - outs[0]).max() <= 1e-3


def test_lse_output(cuda):
    p = W.workload("gqa4_b4_paged", shrink=8, n_layers=1, steps=1)
    for S in (1, 6):
        ws = Workspace.from_problem(p, max_splits=S)
        run = DecodeRunner(ws, p.batch, num_splits=S, flags=A.PKV_FLAG_WRITE_LSE, scale=p.scale)
        q, k, v = W.step_inputs(p, 0)
        run.q_in.copy_(q), run.k_in.copy_(k), run.v_in.copy_(v)
        run.step()
        torch.cuda.synchronize()
        from parity import OracleState
        st = OracleState(p)
        st.bind()
        st.append(0, R.tensor_bits(k)[0], R.tensor_bits(v)[0])
        _, lse = st.attention(0, R.tensor_bits(q)[0])
        assert np.abs(ws.lse[:p.batch].cpu().numpy() - lse).max() <= 1e-3


@pytest.mark.parametrize("fused", [False, True])
def test_graph_replay_bitexact(cuda, fused):
    # A captured step replays to exactly the eager result (same kernels, same plan).
    p = W.workload("gqa8_graph_sweep", batch=8, shrink=16, steps=1)
    q, k, v = W.step_inputs(p, 0)
    res = []
    for use_graph in (False, True):
        ws = Workspace.from_problem(p, max_splits=4)
        run = DecodeRunner(ws, p.batch, num_splits=4, scale=p.scale, fused=fused)
        run.q_in.copy_(q), run.k_in.copy_(k), run.v_in.copy_(v)
        if use_graph:
            run.capture()
            torch.cuda.synchronize()
            assert ws.seq_lens[:p.batch].tolist() == p.seq_lens.tolist()  # capture ran nothing
            run.replay()
        else:
            run.step()
        torch.cuda.synchronize()
        res.append((ws.out_bf16(p.batch).cpu().clone(), ws.seq_lens[:p.batch].cpu().clone(),
                    ws.kv_indptr[:p.batch + 1].cpu().clone(), ws.k_pool.cpu().clone()))
    for a, b in zip(*res):
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b)


def test_rebuild_after_batch_change(cuda):
    # A changed task set must be rebound with REBUILD from caller-written lengths.
    p = W.workload("gqa4_b4_paged", shrink=16, n_layers=1, steps=4)
    ws = Workspace.from_problem(p, max_splits=2)
    lens = [5, 40, 17, 2]
    ws.seq_lens[:4].copy_(torch.tensor(lens, dtype=torch.int32))
    A.pkv_bind_step(ws, 4, A.PKV_BIND_REBUILD)
    torch.cuda.synchronize()
    ref = R.bind(lens, req_pool_indices=p.req_pool_indices.numpy(),
                 page_table=p.page_table.numpy(), page_size=p.page_size, mode=R.REBUILD)
    assert ws.seq_lens[:4].tolist() == ref["seq_lens"]
    assert ws.position_ids[:4].tolist() == ref["position_ids"]
    assert ws.kv_indptr[:5].tolist() == ref["kv_indptr"]
    assert ws.out_loc[:4].tolist() == ref["out_loc"]


@pytest.mark.parametrize("kern", ["mma", "fused", "fused_gather"])
def test_batch_beyond_compact_plan(cuda, kern):
    # More requests than the blocks plan compactly (256): every unit is
    # enumerated, splits of requests shorter than the chunk are empty.
    rng = np.random.default_rng(11)
    lens = [int(x) for x in rng.integers(1, 97, size=300)]
    lens[5] = 0
    p = W.make_problem("wide", batch=300, n_layers=1, n_q_heads=8, n_kv_heads=2, head_dim=64,
                       page_size=16, seq_lens=lens, steps=1, seed=12)
    run_steps(p, S=3, heads=_sample_heads(p, 40), check_partials=True, check_pool=True,
              flags=PATHS[kern][0], fused=PATHS[kern][1])


def test_zero_length_request(cuda):
    # A request with no tokens gives zeros (and lse = -inf), with no error bit.
    p = W.make_problem("zero", batch=3, n_layers=1, n_q_heads=8, n_kv_heads=2, head_dim=128,
                       page_size=16, seq_lens=[10, 0, 50], seed=4)
    for S, fused in ((1, False), (3, False), (1, True), (3, True)):
        ws = Workspace.from_problem(p, max_splits=S)
        q = W.normal_bf16((3, 8, 128), 5).to("cuda")
        A.pkv_bind_step(ws, 3, A.PKV_BIND_REBUILD)
        if fused:
            A.pkv_decode_layer(ws, 3, 0, q, None, None, p.scale, S, A.PKV_FLAG_WRITE_LSE)
        else:
            A.pkv_decode_attn(ws, 3, 0, q, p.scale, S, A.PKV_FLAG_WRITE_LSE)
            A.pkv_merge_partials(ws, 3, S, A.PKV_FLAG_WRITE_LSE)
        torch.cuda.synchronize()
        out = bf16_to_f64(ws.out_bf16(3))
        assert np.all(out[1] == 0) and np.all(np.isneginf(ws.lse[1].cpu().numpy()))
        assert int(ws.err.item()) == 0
        st_slots = [R.token_slots(b, L, page_table=p.page_table.numpy(),
                                  req_pool_indices=p.req_pool_indices.numpy(), page_size=16)
                    for b, L in enumerate([10, 0, 50])]
        ref, _ = R.decode_attention(R.tensor_bits(q.cpu()), R.tensor_bits(p.k_pool),
                                    R.tensor_bits(p.v_pool), 0, st_slots, p.scale, 2)
        check_attention(out, ref, f"zero-length S={S}")


# ----------------------------------------------------------- full size ----

def _bench_splits(p, chooser=A.pkv_choose_splits):
    ws_shape = A.PkvWorkspace(n_kv_heads=p.n_kv_heads, max_splits=256)
    return chooser(ws_shape, p.batch, int(p.seq_lens.max()) + 1,
                   int(p.seq_lens.sum()) + p.batch, _sms())


@pytest.mark.parametrize("name,batch", [("gqa4_b4_paged", None), ("gqa4_b16_flat_skewed", None),
                                        ("gqa4_long_65536", 1), ("gqa4_long_65536", 4),
                                        ("gqa8_graph_sweep", 16), ("gqa8_graph_sweep", 32),
                                        ("gqa8_graph_sweep", 64)])
def test_full_size_sampled(cuda, name, batch):
    p = W.workload(name, batch=batch, steps=1)
    layers = sorted({0, p.n_layers - 1})
    # the fused layer kernel the benchmark times (apportioned splits, S from
    # pkv_choose_pieces), then the unfused tensor-core path
    for flags, fused, chooser in ((0, True, A.pkv_choose_pieces),
                                  (MMA, False, A.pkv_choose_splits)):
        S = _bench_splits(p, chooser)
        run_steps(p, S=S, check_layers=layers, heads=_sample_heads(p, 12), check_partials=True,
                  flags=flags, fused=fused)


def test_kernels_agree(cuda):
    # fp32 outputs of the CUDA-core and both tensor-core producers, same inputs.
    p = W.workload("gqa8_graph_sweep", batch=4, shrink=8, steps=1)
    outs = []
    for kern in (SIMT, MMA, MMA | GATHER):
        ws = Workspace.from_problem(p, max_splits=3)
        run = DecodeRunner(ws, p.batch, num_splits=3, flags=kern | A.PKV_FLAG_OUT_F32,
                           scale=p.scale)
        q, k, v = W.step_inputs(p, 0)
        run.q_in.copy_(q), run.k_in.copy_(k), run.v_in.copy_(v)
        run.step()
        torch.cuda.synchronize()
        outs.append(ws.out_f32(p.batch).cpu().numpy())
    assert np.abs(outs[0] - outs[1]).max() <= 1e-3
    assert np.abs(outs[0] - outs[2]).max() <= 1e-3


# ------------------------------------------------------------ step plan ----

def _fused_out(p, S, flags=0, plan=True, plan_args=None):
    ws = Workspace.from_problem(p, max_splits=max(S, 8))
    run = DecodeRunner(ws, p.batch, num_splits=S, flags=flags | A.PKV_FLAG_OUT_F32,
                       scale=p.scale, plan=plan)
    q, k, v = W.step_inputs(p, 0)
    run.q_in.copy_(q), run.k_in.copy_(k), run.v_in.copy_(v)
    if plan_args is not None:
        # a plan made for other arguments: the layers must ignore it
        A.pkv_bind_step(ws, p.batch, A.PKV_BIND_STEADY, 0, 0, None, None)
        A.pkv_plan_step(ws, *plan_args)
        for l in range(p.n_layers):
            A.pkv_decode_layer(ws, p.batch, l, run.q_in[l], run.k_in[l], run.v_in[l], p.scale,
                               S, flags | A.PKV_FLAG_OUT_F32 | A.PKV_FLAG_USE_PLAN)
    else:
        run.step()
    torch.cuda.synchronize()
    assert int(ws.err.item()) == 0
    assert int(ws.split_counters.abs().sum().item()) == 0
    return ws.out_f32(p.batch).cpu().numpy().copy()


@pytest.mark.parametrize("name,batch", [("gqa4_b4_paged", None), ("gqa8_graph_sweep", 16),
                                        ("gqa4_b16_flat_skewed", None)])
def test_step_plan_bitexact(cuda, name, batch):
    # Layers that read the step's plan compute exactly what layers that plan
    # for themselves compute (same splits, same arithmetic).
    p = W.workload(name, batch=batch, shrink=4, steps=1)
    S = _bench_splits(p, A.pkv_choose_pieces)
    a = _fused_out(p, S, plan=True)
    b = _fused_out(p, S, plan=False)
    assert np.array_equal(a, b)


def test_step_plan_for_other_arguments_is_ignored(cuda):
    p = W.workload("gqa4_b4_paged", shrink=8, steps=1)
    ref = _fused_out(p, 4, plan=False)
    for other in ((p.batch, 3, 0), (p.batch - 1, 4, 0), (p.batch, 4, A.PKV_FLAG_FIXED_CHUNK),
                  (p.batch, 4, A.PKV_FLAG_FORCE_GATHER)):
        got = _fused_out(p, 4, plan_args=other)
        assert np.array_equal(got, ref), other


# ------------------------------------------------------ token-level pages ----

@pytest.mark.parametrize("D,G,Hkv,P", [(128, 4, 8, 1), (128, 2, 4, 1), (64, 1, 4, 1),
                                       (64, 4, 8, 8), (128, 1, 8, 1)])
@pytest.mark.parametrize("S", [1, 3])
def test_token_level_variants(cuda, D, G, Hkv, P, S):
    # Flat token-level indices and pages shorter than a 16-token box, over head
    # dims, group sizes and KV head counts: the fused layer's gather producer
    # (and the flat bind / append around it).
    rng = np.random.default_rng(D + G + Hkv + P)
    lens = [int(x) for x in rng.integers(1, 300, size=5)]
    p = W.make_problem("rows", batch=5, n_layers=2, n_q_heads=G * Hkv, n_kv_heads=Hkv,
                       head_dim=D, page_size=P, seq_lens=lens, steps=1, seed=13)
    run_steps(p, S=S, check_pool=True, fused=True)


# ------------------------------------------------- cache layouts (next) ----

@pytest.mark.parametrize("P", [2048, 1040])
def test_contiguous_cache(cuda, P):
    # One page per request holding its whole context (page size = capacity):
    # a contiguous cache as a special case of the page table.  1040 is a
    # multiple of 16 but no power of two (the page arithmetic divides).
    lens = [1500, 7, 1023, 2000] if P == 2048 else [1000, 7, 1023, 640]
    p = W.make_problem("contig", batch=4, n_layers=1, n_q_heads=16, n_kv_heads=4,
                       head_dim=128, page_size=P, seq_lens=lens, steps=1, seed=21)
    assert p.max_pages_per_req == 1
    for S, kern in ((1, "fused"), (4, "fused"), (4, "mma"), (4, "fused_gather")):
        run_steps(p, S=S, check_pool=True, check_partials=kern == "mma",
                  flags=PATHS[kern][0], fused=PATHS[kern][1])


def test_shared_prefix_pages(cuda):
    # Requests whose tables alias the same physical pages for a common prefix
    # (each appends into a page of its own): every request attends to the
    # shared prefix's K/V.
    lens = [200, 150, 180, 170]
    p = W.make_problem("prefix", batch=4, n_layers=2, n_q_heads=16, n_kv_heads=4,
                       head_dim=128, page_size=16, seq_lens=lens, steps=1, seed=22)
    rows = p.req_pool_indices.tolist()
    shared = p.page_table[rows[0], :5].clone()
    for b in range(1, 4):
        p.page_table[rows[b], :5] = shared
    for kern in ("fused", "mma", "fused_gather"):
        run_steps(p, S=3, check_pool=True, check_partials=kern == "mma",
                  flags=PATHS[kern][0], fused=PATHS[kern][1])


def test_shared_prefix_workload_small(cuda):
    # The benchmark's prefix-shared workload (every request's first pages are
    # one set stored once), oracle-sized: fused decode through the aliased pages.
    p = W.workload("shared_prefix_b32", shrink=16, steps=1)
    run_steps(p, S=4, check_pool=True)


# ------------------------------------------- the block-wide batch plan ----

_PLAN_PROBLEMS = {}


@pytest.mark.parametrize("plan", [False, True], ids=["self_planned", "step_plan"])
@pytest.mark.parametrize("producer", ["tma", "gather"])
@pytest.mark.parametrize("B", [33, 64, 200])
def test_block_wide_plan_batches(cuda, B, producer, plan):
    # 33..256 requests: the fused layer's compact plan runs its block-wide
    # scan (one warp plans up to 32 requests), with the step's plan and
    # without, for both producers; every output element is compared.
    if B not in _PLAN_PROBLEMS:
        _PLAN_PROBLEMS[B] = W.workload("gqa8_graph_sweep", batch=B, shrink=16, steps=1)
    p = _PLAN_PROBLEMS[B]
    assert 32 < p.batch <= 256
    run_steps(p, S=4, check_pool=True, flags=GATHER if producer == "gather" else 0, fused=True,
              plan=plan)


# --------------------------------------------- REBUILD at large batch ----

@pytest.mark.parametrize("B", [64, 256, 2000])
def test_rebuild_changed_task_set_large_batch(cuda, B):
    # A steady step, then the task set changes (a quarter of the requests
    # leave, the rest come back in another order, each one token longer): the
    # host sees a non-steady step, writes the lengths and request rows, and
    # the REBUILD bind and a fused layer follow.  Metadata bit-exact, the
    # appended pool bit-exact, attention against the oracle (sampled heads
    # for the largest batch).  2000 requests take the bind kernel's
    # several-requests-per-thread scan and the fused layer's enumeration
    # without the compact plan.
    rng = np.random.default_rng(B)
    lens = [int(x) for x in rng.integers(1, 97, size=B)]
    p = W.make_problem("rebuild", batch=B, n_layers=1, n_q_heads=8, n_kv_heads=2, head_dim=64,
                       page_size=16, seq_lens=lens, steps=2, seed=40 + B)
    S = 3
    ws = Workspace.from_problem(p, max_splits=S)
    tracker = BindTracker()
    ids = list(range(B))
    assert tracker.mode(ids, lens) == A.PKV_BIND_REBUILD  # the first bind
    heads = _sample_heads(p, 64) if B > 256 else None
    # step 0: steady (every length + 1)
    assert tracker.mode(ids, [x + 1 for x in lens]) == A.PKV_BIND_STEADY
    run = DecodeRunner(ws, B, num_splits=S, scale=p.scale)
    q, k, v = W.step_inputs(p, 0)
    run.q_in.copy_(q), run.k_in.copy_(k), run.v_in.copy_(v)
    run.step()
    st = OracleState(p)
    st.bind()
    st.append(0, R.tensor_bits(k)[0], R.tensor_bits(v)[0])
    torch.cuda.synchronize()
    check_meta(ws, st, B)
    # step 1: a changed task set
    keep = rng.permutation(B)[: B - B // 4]
    B2 = len(keep)
    new_ids = [ids[i] for i in keep]
    new_lens = [st.lens[i] + 1 for i in keep]
    new_rows = p.req_pool_indices.numpy()[keep]
    assert tracker.mode(new_ids, new_lens) == A.PKV_BIND_REBUILD
    ws.seq_lens[:B2].copy_(torch.tensor(new_lens, dtype=torch.int32))
    ws.req_pool_indices[:B2].copy_(torch.from_numpy(new_rows.astype(np.int32)))
    run2 = DecodeRunner(ws, B2, num_splits=S, scale=p.scale)
    q2 = W.normal_bf16((1, B2, 8, 64), 7000 + B)
    k2 = W.normal_bf16((1, B2, 2, 64), 7001 + B)
    v2 = W.normal_bf16((1, B2, 2, 64), 7002 + B)
    run2.q_in.copy_(q2), run2.k_in.copy_(k2), run2.v_in.copy_(v2)
    run2.step(A.PKV_BIND_REBUILD)
    torch.cuda.synchronize()
    assert int(ws.err.item()) == 0
    assert int(ws.split_counters.abs().sum().item()) == 0
    table = p.page_table.numpy()
    meta = R.bind(new_lens, req_pool_indices=new_rows, page_table=table, page_size=16,
                  mode=R.REBUILD)
    assert ws.seq_lens[:B2].tolist() == meta["seq_lens"]
    assert ws.position_ids[:B2].tolist() == meta["position_ids"]
    assert ws.kv_indptr[:B2 + 1].tolist() == meta["kv_indptr"]
    assert ws.out_loc[:B2].tolist() == meta["out_loc"]
    kb = R.append_rows(st.kb, 0, meta["out_loc"], R.tensor_bits(k2)[0])
    vb = R.append_rows(st.vb, 0, meta["out_loc"], R.tensor_bits(v2)[0])
    assert np.array_equal(R.tensor_bits(ws.k_pool.cpu()), kb)
    assert np.array_equal(R.tensor_bits(ws.v_pool.cpu()), vb)
    slots = [R.token_slots(b, meta["seq_lens"][b], page_table=table, req_pool_indices=new_rows,
                           page_size=16) for b in range(B2)]
    heads2 = None if heads is None else [(b, h) for b, h in heads if b < B2]
    ref, _ = R.decode_attention(R.tensor_bits(q2)[0], kb, vb, 0, slots, p.scale, 2,
                                heads=heads2)
    got = bf16_to_f64(ws.out_bf16(B2))
    if heads2 is not None:
        idx = tuple(np.array(heads2).T)
        got, ref = got[idx], ref[idx]
    check_attention(got, ref, f"REBUILD B={B} -> {B2}")
