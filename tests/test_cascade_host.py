"""Host logic of CascadeDecoder and DecodeRunner on a CPU workspace (nothing
is launched): the cascade's argument checks, its two views over the
workspace and its split rule, and the runner's kernel count per step."""
import pytest
import torch

from paged_kv_decode_bind_gb300 import CascadeDecoder, Workspace, choose_prefix_splits
from paged_kv_decode_bind_gb300 import _abi as A


def _ws(page_size=16, max_splits=4):
    ws = Workspace(n_layers=2, pool_slots=64 * page_size, n_q_heads=8, n_kv_heads=2,
                   head_dim=64, page_size=page_size, max_batch=4, max_reqs=4,
                   max_pages_per_req=16, max_splits=max_splits, max_total_tokens=1024,
                   device="cpu")
    ws.seq_lens[:3] = torch.tensor([70, 90, 64], dtype=torch.int32)
    ws.req_pool_indices[:3] = torch.tensor([2, 0, 1], dtype=torch.int32)
    return ws


def test_rejects_a_prefix_that_is_not_whole_pages():
    with pytest.raises(ValueError):
        CascadeDecoder(_ws(), 3, 40, scale=0.125)


def test_rejects_flat_indices():
    with pytest.raises(ValueError):
        CascadeDecoder(_ws(page_size=1), 3, 32, scale=0.125)


def test_rejects_more_suffix_splits_than_the_workspace_holds():
    with pytest.raises(ValueError):
        CascadeDecoder(_ws(max_splits=2), 3, 32, scale=0.125, suffix_splits=3)


def test_views():
    ws = _ws()
    cas = CascadeDecoder(ws, 3, 48, scale=0.125, prefix_splits=2)
    vp, vs = cas.prefix_view, cas.suffix_view
    # prefix: one request, request 0's page-table row, prefix_len tokens; its
    # batch * Hq query rows get lse rows and, with splits, partials of their own
    assert vp.seq_lens == cas.prefix_lens.data_ptr() and cas.prefix_lens.tolist() == [48]
    assert cas.prefix_row.tolist() == [2]
    assert vp.max_batch == 3 and vp.max_splits == 2
    assert vp.lse == cas.lse_prefix.data_ptr() and cas.lse_prefix.numel() == 3 * 8
    assert cas.part_o.numel() == 3 * 8 * 2 * 64 and cas.part_ml.numel() == 3 * 8 * 2 * 2
    assert cas.qo_indptr.tolist() == [0, 3]
    # suffix: the table from the first page past the prefix, the own lengths,
    # private bind outputs; the main workspace's pointers are untouched
    assert vs.page_table == ws.page_table.data_ptr() + 3 * 4
    assert vs.seq_lens == cas.suffix_lens.data_ptr()
    assert cas.suffix_lens.tolist() == [22, 42, 16]
    assert vs.kv_indptr == cas.suffix_indptr.data_ptr()
    assert vs.position_ids == cas.suffix_positions.data_ptr()
    assert vs.out_loc == cas.suffix_out_loc.data_ptr()
    assert vs.out == cas.out_suffix.data_ptr() and vs.lse == cas.lse_suffix.data_ptr()
    assert vs.req_pool_indices == ws.struct.req_pool_indices
    assert ws.struct.page_table == ws.page_table.data_ptr()
    assert ws.struct.seq_lens == ws.seq_lens.data_ptr()
    # both views keep the pools and the model shape
    for v in (vp, vs):
        assert v.k_pool == ws.struct.k_pool and v.v_pool == ws.struct.v_pool
        assert (v.n_q_heads, v.n_kv_heads, v.head_dim, v.page_size) == (8, 2, 64, 16)
        assert v.index_mode == A.PKV_IDX_PAGE_TABLE


def test_rejects_zero_splits():
    with pytest.raises(ValueError):
        CascadeDecoder(_ws(), 3, 32, scale=0.125, prefix_splits=0)


def test_choose_prefix_splits():
    # 32 requests, G = 4: 16 per block, 2 blocks per KV head, 16 blocks; two
    # per SM on 152 SMs leave room for 19 splits, and a 4096-token prefix
    # allows 16 of at least 256 keys
    assert choose_prefix_splits(32, 4, 8, 4096, 152) == 16
    assert choose_prefix_splits(32, 4, 8, 4096 * 4, 152) == 19
    # short prefixes are not split; G = 16 packs 4 requests in a block: 8
    # blocks per KV head, 16 blocks over 2 KV heads
    assert choose_prefix_splits(32, 4, 8, 255, 152) == 1
    assert choose_prefix_splits(32, 16, 2, 65536, 152) == 19
    # more blocks than two per SM: one split
    assert choose_prefix_splits(4096, 1, 8, 65536, 152) == 1


def test_decode_runner_launch_count():
    # kernels per step, as the bench reports them: the bind (+ the flat index
    # build), then per layer one fused kernel, or append + attention (+ merge
    # when split); the step's plan adds one launch when used
    from paged_kv_decode_bind_gb300 import DecodeRunner
    ws = _ws()  # 2 layers, G = 4, D = 64, page table
    assert DecodeRunner(ws, 3, num_splits=4).launches_per_step == 1 + 2
    assert DecodeRunner(ws, 3, num_splits=4, fused=False).launches_per_step == 1 + 2 * 3
    assert DecodeRunner(ws, 3, num_splits=1, fused=False).launches_per_step == 1 + 2 * 2
    simt = DecodeRunner(ws, 3, num_splits=4, flags=A.PKV_FLAG_FORCE_SIMT)
    assert simt.launches_per_step == 1 + 2 * 3  # no fused CUDA-core kernel
    assert DecodeRunner(ws, 3, num_splits=4, plan=True).launches_per_step == 1 + 1 + 2
    flat = _ws(page_size=1)
    assert DecodeRunner(flat, 3, num_splits=4).launches_per_step == 2 + 2


def test_rejects_batch_beyond_the_workspace():
    # the suffix pass writes batch * Hq * S partial rows into the workspace's
    # o_part / ml_part and reads batch entries of its request rows
    with pytest.raises(ValueError):
        CascadeDecoder(_ws(), 5, 32, scale=0.125)  # max_batch is 4
    with pytest.raises(ValueError):
        CascadeDecoder(_ws(), 0, 32, scale=0.125)
    assert CascadeDecoder(_ws(), 4, 32, scale=0.125).suffix_view.max_batch == 4


def test_suffix_length_limit():
    # rows of 16 pages of 16 tokens; a 48-token prefix leaves 13 pages for
    # the suffix: the view keeps the table's row stride (16 entries) and
    # limits the suffix length to 13 * 16, which the device checks
    ws = _ws()
    vs = CascadeDecoder(ws, 3, 48, scale=0.125).suffix_view
    assert vs.max_pages_per_req == 16
    assert vs.max_seq_len == 13 * 16
    assert ws.struct.max_seq_len == 0  # the main workspace: the whole row
    # the boundary: a prefix of 15 pages leaves one page, 16 pages none
    assert CascadeDecoder(ws, 3, 15 * 16, scale=0.125).suffix_view.max_seq_len == 16
    with pytest.raises(ValueError):
        CascadeDecoder(ws, 3, 16 * 16, scale=0.125)


def test_prefix_kernel_choice():
    # The prefix pass takes the tcgen05 extend kernel from 512 prefix tokens a
    # split, the warp-level one below (its units too short for the 128-row
    # CTAs' setup)
    ws = Workspace(n_layers=1, pool_slots=512 * 16, n_q_heads=8, n_kv_heads=2, head_dim=64,
                   page_size=16, max_batch=4, max_reqs=4, max_pages_per_req=512,
                   max_splits=16, max_total_tokens=8192, device="cpu")
    ws.req_pool_indices[:2] = torch.tensor([0, 1], dtype=torch.int32)
    ws.seq_lens[:2] = torch.tensor([4200, 4300], dtype=torch.int32)
    for splits, kernel in [(1, 0), (8, 0), (9, A.PKV_FLAG_EXTEND_WARP_MMA),
                           (16, A.PKV_FLAG_EXTEND_WARP_MMA)]:
        cas = CascadeDecoder(ws, 2, 4096, scale=0.125, prefix_splits=splits)
        assert cas.prefix_kernel == kernel, splits
