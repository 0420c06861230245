"""Device-side error handling: invalid indices are caught by the kernels' own
bounds checks before any access, raise their bit in the sticky err word and
leave finite outputs; the other requests of the batch stay correct.

Every invalid value used here is one the kernels check (page ids against the
pool, slots against the pool, lengths against the table capacity, table rows
against max_reqs), so nothing here can fault the GPU.
"""
import numpy as np
import pytest
import torch

import oracle.ref as R
import pkv_inputs as W
from paged_kv_decode_bind_gb300 import DecodeRunner, Workspace
from paged_kv_decode_bind_gb300 import _abi as A

from parity import OracleState, bf16_to_f64, check_attention

pytestmark = pytest.mark.gpu

PATHS = {"simt": (A.PKV_FLAG_FORCE_SIMT, False), "mma": (A.PKV_FLAG_FORCE_MMA, False),
         "gather": (A.PKV_FLAG_FORCE_MMA | A.PKV_FLAG_FORCE_GATHER, False),
         "fused": (0, True), "fused_gather": (A.PKV_FLAG_FORCE_GATHER, True),
         "fused_fixed": (A.PKV_FLAG_FIXED_CHUNK, True)}


def _setup(p, S, kern):
    flags, fused = PATHS[kern]
    ws = Workspace.from_problem(p, max_splits=S)
    run = DecodeRunner(ws, p.batch, num_splits=S, flags=flags, scale=p.scale, fused=fused)
    q, k, v = W.step_inputs(p, 0)
    run.q_in.copy_(q), run.k_in.copy_(k), run.v_in.copy_(v)
    return ws, run, q, k, v


def _check_others(p, ws, q, k, v, bad_b, layer=0):
    st = OracleState(p)
    st.bind()
    st.append(layer, R.tensor_bits(k)[layer], R.tensor_bits(v)[layer])
    heads = [(b, h) for b in range(p.batch) if b != bad_b for h in range(p.n_q_heads)]
    ref, _ = st.attention(layer, R.tensor_bits(q)[layer], heads=heads)
    got = bf16_to_f64(ws.out_bf16(p.batch))
    idx = tuple(np.array(heads).T)
    check_attention(got[idx], ref[idx], "healthy requests")
    assert np.all(np.isfinite(got))


@pytest.mark.parametrize("kern", list(PATHS))
@pytest.mark.parametrize("S", [1, 3])
def test_bad_page_id(cuda, kern, S):
    p = W.workload("gqa4_b4_paged", shrink=8, n_layers=1, steps=1)
    ws, run, q, k, v = _setup(p, S, kern)
    row = int(p.req_pool_indices[1])
    n_pages = p.pool_slots // p.page_size
    ws.page_table[row, 0] = n_pages + 5  # first page of request 1 out of range
    run.step()
    torch.cuda.synchronize()
    assert int(ws.err.item()) & A.PKV_DEVERR_PAGE
    # the other requests' pages are untouched, so the oracle keeps the
    # original table for them
    _check_others(p, ws, q, k, v, bad_b=1)


@pytest.mark.parametrize("kern", list(PATHS))
def test_length_over_capacity(cuda, kern):
    p = W.workload("gqa4_b4_paged", shrink=8, n_layers=1, steps=1)
    ws, run, q, k, v = _setup(p, 2, kern)
    cap = p.max_pages_per_req * p.page_size
    lens = p.seq_lens.tolist()
    lens[2] = cap + 5
    ws.seq_lens[:p.batch].copy_(torch.tensor(lens, dtype=torch.int32))
    run.bind(A.PKV_BIND_REBUILD)
    for l in range(p.n_layers):
        run.layer(l)
    torch.cuda.synchronize()
    assert int(ws.err.item()) & A.PKV_DEVERR_LEN
    out = bf16_to_f64(ws.out_bf16(p.batch))
    assert np.all(np.isfinite(out)) and np.all(out[2] == 0)


@pytest.mark.parametrize("kern", ["simt", "gather", "fused"])
def test_flat_bad_slot(cuda, kern):
    p = W.workload("gqa4_b16_flat_skewed", shrink=16, n_layers=1, steps=1)
    ws, run, q, k, v = _setup(p, 2, kern)
    run.bind()
    # corrupt one token's slot of request 0 after the bind built kv_indices
    ws.kv_indices[0] = p.pool_slots + 3
    for l in range(p.n_layers):
        run.layer(l)
    torch.cuda.synchronize()
    assert int(ws.err.item()) & A.PKV_DEVERR_SLOT
    assert np.all(np.isfinite(bf16_to_f64(ws.out_bf16(p.batch))))


@pytest.mark.parametrize("kern", ["simt", "mma", "fused"])
def test_bad_table_row(cuda, kern):
    p = W.workload("gqa4_b4_paged", shrink=8, n_layers=1, steps=1)
    ws, run, q, k, v = _setup(p, 3, kern)
    ws.req_pool_indices[3] = -7
    run.step()
    torch.cuda.synchronize()
    assert int(ws.err.item()) & A.PKV_DEVERR_PAGE
    assert np.all(np.isfinite(bf16_to_f64(ws.out_bf16(p.batch))))


def test_err_word_is_sticky_and_cleared_by_caller(cuda):
    p = W.workload("gqa4_b4_paged", shrink=8, n_layers=1, steps=2)
    ws, run, q, k, v = _setup(p, 1, "fused")
    ws.req_pool_indices[0] = 10 ** 6
    run.step()
    torch.cuda.synchronize()
    assert int(ws.err.item()) != 0
    ws.err.zero_()
    ws.req_pool_indices[0] = int(p.req_pool_indices[0])
    ws.seq_lens[:p.batch].copy_(p.seq_lens)
    run.step()
    torch.cuda.synchronize()
    assert int(ws.err.item()) == 0


@pytest.mark.parametrize("kern", ["fused", "fused_gather"])
def test_bounded_wait_runs_out(cuda, kern):
    # The test hook leaves every block's first tile unloaded, so the
    # consumers' bounded wait for it runs out (~1 s): the launch sets
    # PKV_DEVERR_TIMEOUT and returns with empty (finite) outputs and its split
    # counters back at zero, and the context stays usable.
    from parity import run_steps
    p = W.workload("gqa4_b4_paged", shrink=8, n_layers=1, steps=1)
    ws, run, q, k, v = _setup(p, 2, kern)
    run.bind()
    A.pkv_decode_layer(ws, p.batch, 0, run.q_in[0], run.k_in[0], run.v_in[0], p.scale, 2,
                       PATHS[kern][0] | A.PKV_FLAG_TEST_SKIP_FIRST_TILE)
    torch.cuda.synchronize()
    assert int(ws.err.item()) & A.PKV_DEVERR_TIMEOUT
    assert np.all(np.isfinite(bf16_to_f64(ws.out_bf16(p.batch))))
    assert int(ws.split_counters.abs().sum().item()) == 0
    run_steps(p, S=2, flags=PATHS[kern][0], fused=True)  # a normal launch afterwards
