"""Decode attention for a batch whose requests share prefix pages.

When every request of a batch starts with the same ``prefix_len`` tokens
stored in the same physical pages (the engine's prefix-shared pages: many
requests aliasing one prompt's pages), attending each request's whole
context reads the shared prefix once per request.  ``CascadeDecoder`` reads
it once for the batch, in three calls of the C ABI per layer:

1. ``pkv_extend_attn`` with ``PKV_FLAG_EXTEND_FULL`` over a one-request view
   of the workspace whose context is the prefix: every (request, query head)
   row attends all ``prefix_len`` tokens, writing its normalised output and
   log-sum-exp;
2. ``pkv_decode_attn`` over a view whose page table starts past the prefix's
   pages and whose lengths are the requests' own suffix lengths;
3. ``pkv_merge_lse``, which combines the two by log-sum-exp into ``out``.

Every buffer is allocated here once, at fixed addresses, so a step (and its
capture into a CUDA graph) allocates nothing.  The suffix lengths live in
``suffix_lens``; ``bind`` advances them with the library's metadata bind on
the suffix view (and appends the new K/V rows), like ``pkv_bind_step`` does
for a plain batch; the view has its own ``kv_indptr``, ``position_ids`` and
``out_loc`` (positions relative to the end of the prefix), so the main
workspace's metadata is left as it is.
"""
from __future__ import annotations

import torch

from . import _abi


def choose_prefix_splits(batch: int, group: int, n_kv_heads: int, prefix_len: int,
                         num_sms: int) -> int:
    """Splits of the shared prefix for the extend kernel's pass over it: as
    many as keep its blocks within one wave of two per SM, and no split
    shorter than four 64-key tiles.  A block holds 64 query rows, 64 / group
    requests of one KV head."""
    per_block = max(1, 64 // group)
    blocks = -(-batch // per_block) * n_kv_heads
    return max(1, min(2 * num_sms // max(1, blocks), prefix_len // 256))


class CascadeDecoder:
    def __init__(self, ws, batch: int, prefix_len: int, *, scale: float, prefix_splits: int = 1,
                 suffix_splits: int = 1):
        sh = ws.shape
        P, Hq, D = sh["page_size"], sh["n_q_heads"], sh["head_dim"]
        if sh["index_mode"] != _abi.PKV_IDX_PAGE_TABLE or prefix_len % P:
            raise ValueError("the shared prefix must be whole pages of a page-table workspace")
        if suffix_splits > sh["max_splits"]:
            raise ValueError("suffix_splits exceeds the workspace's max_splits")
        if prefix_splits < 1 or suffix_splits < 1:
            raise ValueError("split counts start at 1")
        if not 0 < batch <= sh["max_batch"]:
            raise ValueError("batch must be in 1 .. the workspace's max_batch")
        # the suffix view's rows start prefix_len / P entries into the table's
        # rows: they keep the table's stride but hold only the rest of a row
        suffix_cap = (sh["max_pages_per_req"] - prefix_len // P) * P
        if suffix_cap <= 0:
            raise ValueError("the shared prefix fills the whole page-table row")
        dev = ws.device
        f32 = dict(dtype=torch.float32, device=dev)
        i32 = dict(dtype=torch.int32, device=dev)
        self.ws, self.batch, self.prefix_len, self.scale = ws, batch, prefix_len, scale
        self.prefix_splits, self.suffix_splits = prefix_splits, suffix_splits
        self.out_prefix = torch.zeros((batch, Hq, D), **f32)
        self.out_suffix = torch.zeros((batch, Hq, D), **f32)
        self.lse_prefix = torch.zeros(batch * Hq, **f32)
        self.lse_suffix = torch.zeros(batch * Hq, **f32)
        self.qo_indptr = torch.tensor([0, batch], **i32)
        self.prefix_lens = torch.tensor([prefix_len], **i32)
        self.prefix_row = ws.req_pool_indices[:1].clone()
        self.part_o = torch.zeros(batch * Hq * max(1, prefix_splits) * D, **f32)
        self.part_ml = torch.zeros(batch * Hq * max(1, prefix_splits) * 2, **f32)
        self.suffix_lens = (ws.seq_lens[:batch] - prefix_len).contiguous()
        self.suffix_indptr = torch.zeros(batch + 1, **i32)
        self.suffix_positions = torch.zeros(batch, **i32)
        self.suffix_out_loc = torch.zeros(batch, **i32)
        # prefix view: one request (request 0's table row) of prefix_len tokens
        # whose batch's queries are the extend rows
        vp = _abi.PkvWorkspace.from_buffer_copy(ws.struct)
        vp.seq_lens, vp.req_pool_indices = self.prefix_lens.data_ptr(), self.prefix_row.data_ptr()
        vp.max_batch, vp.max_splits = batch, max(1, prefix_splits)
        vp.lse, vp.o_part, vp.ml_part = (self.lse_prefix.data_ptr(), self.part_o.data_ptr(),
                                         self.part_ml.data_ptr())
        self.prefix_view = vp
        # suffix view: the table past the prefix's pages, the own lengths
        vs = _abi.PkvWorkspace.from_buffer_copy(ws.struct)
        vs.page_table = ws.page_table.data_ptr() + (prefix_len // P) * 4
        vs.seq_lens = self.suffix_lens.data_ptr()
        vs.kv_indptr, vs.position_ids = (self.suffix_indptr.data_ptr(),
                                         self.suffix_positions.data_ptr())
        vs.out_loc = self.suffix_out_loc.data_ptr()
        vs.max_batch = batch  # <= the workspace's: o_part / ml_part hold its rows
        # a suffix length past the rest of the row raises PKV_DEVERR_LEN on the
        # device (the bind and the kernels) instead of reading the next row
        vs.max_seq_len = suffix_cap
        vs.out, vs.lse = self.out_suffix.data_ptr(), self.lse_suffix.data_ptr()
        self.suffix_view = vs
        # The prefix pass's kernel: the tcgen05 one (128-row CTAs, one per SM)
        # spends a few microseconds per unit setting up, so with splits of
        # under 512 prefix tokens the warp-level kernel's 64-row blocks finish
        # first (measured on 32 requests sharing 4096 tokens: 26.2 against
        # 30.2 us per layer with 16 splits of 256; 30.3 and 31.7 with 8)
        self.prefix_kernel = (0 if prefix_len // prefix_splits >= 512
                              else _abi.PKV_FLAG_EXTEND_WARP_MMA)
        # fork / join of the optional second stream (a parallel graph branch)
        self.fork = torch.cuda.Event()
        self.join = torch.cuda.Event()

    def bind(self, mode=_abi.PKV_BIND_STEADY, layer_begin=0, layer_count=0, k_new=None,
             v_new=None, stream=None):
        """Metadata bind (and appends) on the suffix view: its lengths, and
        out_loc of the new tokens past the shared prefix."""
        _abi.pkv_bind_step(self.suffix_view, self.batch, mode, layer_begin, layer_count, k_new,
                           v_new, stream)

    def layer(self, layer, q, out, flags=0, stream=None, suffix_stream=None):
        """Attention of the batch's queries q [batch, Hq, D] over each request's
        shared prefix and own suffix into out (bf16, fp32 with
        PKV_FLAG_OUT_F32).  With suffix_stream the suffix attention runs there,
        concurrently with the prefix's (fork and join by events, which a CUDA
        graph capture turns into a parallel branch)."""
        lse = _abi.PKV_FLAG_OUT_F32 | _abi.PKV_FLAG_WRITE_LSE
        main = stream if stream is not None else torch.cuda.current_stream()
        side = suffix_stream if suffix_stream is not None else main
        if side is not main:
            self.fork.record(main)
            side.wait_event(self.fork)
        _abi.pkv_decode_attn(self.suffix_view, self.batch, layer, q, self.scale,
                             self.suffix_splits, lse, side)
        if self.suffix_splits > 1:
            _abi.pkv_merge_partials(self.suffix_view, self.batch, self.suffix_splits, lse, side)
        _abi.pkv_extend_attn(self.prefix_view, 1, layer, self.qo_indptr, self.batch, q,
                             self.out_prefix, self.scale, num_splits=self.prefix_splits,
                             flags=_abi.PKV_FLAG_EXTEND_FULL | lse | self.prefix_kernel,
                             stream=main)
        if side is not main:
            self.join.record(side)
            main.wait_event(self.join)
        sh = self.ws.shape
        _abi.pkv_merge_lse(self.batch * sh["n_q_heads"], sh["head_dim"], self.out_prefix,
                           self.lse_prefix, self.out_suffix, self.lse_suffix, out, None,
                           flags & _abi.PKV_FLAG_OUT_F32, main)
