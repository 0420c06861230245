"""Caller-owned workspace: torch allocates every buffer once, at fixed device
addresses, and the ctypes ``pkv_workspace`` struct points at them (the
engine's pre-allocated InferenceWorkspace, workspace.py page, bullets 14, 17
and 22).  Nothing in the decode hot loop allocates after construction.
"""
from __future__ import annotations

import torch

from . import _abi


class Workspace:
    """All decode buffers for one model/pool shape.

    ``out`` is allocated with fp32 room so either output type fits; use
    :meth:`out_bf16` / :meth:`out_f32` for typed views.
    """

    def __init__(self, *, n_layers, pool_slots, n_q_heads, n_kv_heads, head_dim, page_size,
                 max_batch, max_reqs, max_pages_per_req, max_splits=1, max_total_tokens=0,
                 index_mode=None, device="cuda", pools=True):
        if index_mode is None:
            index_mode = _abi.PKV_IDX_FLAT if page_size == 1 else _abi.PKV_IDX_PAGE_TABLE
        dev = torch.device(device)
        i32 = dict(dtype=torch.int32, device=dev)
        self.device = dev
        self.shape = dict(n_layers=n_layers, pool_slots=pool_slots, n_q_heads=n_q_heads,
                          n_kv_heads=n_kv_heads, head_dim=head_dim, page_size=page_size,
                          index_mode=index_mode, max_batch=max_batch, max_reqs=max_reqs,
                          max_pages_per_req=max_pages_per_req, max_splits=max_splits,
                          max_total_tokens=max_total_tokens)
        kv_shape = (n_layers, pool_slots, n_kv_heads, head_dim)
        self.k_pool = torch.empty(kv_shape, dtype=torch.bfloat16, device=dev) if pools else None
        self.v_pool = torch.empty(kv_shape, dtype=torch.bfloat16, device=dev) if pools else None
        self.req_pool_indices = torch.zeros(max_batch, **i32)
        self.page_table = torch.full((max_reqs, max_pages_per_req), -1, **i32)
        self.seq_lens = torch.zeros(max_batch, **i32)
        self.position_ids = torch.zeros(max_batch, **i32)
        self.kv_indptr = torch.zeros(max_batch + 1, **i32)
        self.out_loc = torch.zeros(max_batch, **i32)
        self.kv_indices = torch.zeros(max(1, max_total_tokens), **i32)
        self.o_part = torch.zeros((max_batch, n_q_heads, max_splits, head_dim),
                                  dtype=torch.float32, device=dev)
        self.ml_part = torch.zeros((max_batch, n_q_heads, max_splits, 2), dtype=torch.float32,
                                   device=dev)
        self.out = torch.zeros((max_batch, n_q_heads, head_dim), dtype=torch.float32, device=dev)
        self.lse = torch.zeros((max_batch, n_q_heads), dtype=torch.float32, device=dev)
        self.err = torch.zeros(1, **i32)
        self.split_counters = torch.zeros(max(1, max_batch * n_kv_heads), **i32)
        self.work_plan = None  # sized below from the library's layout
        self.struct = _abi.PkvWorkspace(
            **self.shape,
            k_pool=_abi._ptr(self.k_pool) if pools else None,
            v_pool=_abi._ptr(self.v_pool) if pools else None,
            req_pool_indices=self.req_pool_indices.data_ptr(),
            page_table=self.page_table.data_ptr(), seq_lens=self.seq_lens.data_ptr(),
            position_ids=self.position_ids.data_ptr(), kv_indptr=self.kv_indptr.data_ptr(),
            out_loc=self.out_loc.data_ptr(), kv_indices=self.kv_indices.data_ptr(),
            o_part=self.o_part.data_ptr(), ml_part=self.ml_part.data_ptr(),
            out=self.out.data_ptr(), lse=self.lse.data_ptr(), err=self.err.data_ptr(),
            split_counters=self.split_counters.data_ptr())
        plan_bytes = _abi.pkv_workspace_bytes(self.struct, "work_plan")
        self.work_plan = torch.zeros(max(1, plan_bytes // 4), **i32)
        self.struct.work_plan = self.work_plan.data_ptr()

    # typed views of the output buffer --------------------------------------
    def out_bf16(self, batch):
        n = batch * self.shape["n_q_heads"] * self.shape["head_dim"]
        return self.out.view(torch.bfloat16).reshape(-1)[:n].view(
            batch, self.shape["n_q_heads"], self.shape["head_dim"])

    def out_f32(self, batch):
        return self.out[:batch]

    @classmethod
    def from_problem(cls, p, *, max_splits=1, device="cuda", steps_room=0):
        """Workspace sized for a ``pkv_inputs.DecodeProblem`` with its pools,
        table and lengths uploaded."""
        ws = cls(n_layers=p.n_layers, pool_slots=p.pool_slots, n_q_heads=p.n_q_heads,
                 n_kv_heads=p.n_kv_heads, head_dim=p.head_dim, page_size=p.page_size,
                 max_batch=p.batch, max_reqs=p.max_reqs, max_pages_per_req=p.max_pages_per_req,
                 max_splits=max_splits,
                 max_total_tokens=(p.batch * p.max_pages_per_req if p.page_size == 1 else 0),
                 index_mode=p.index_mode, device=device)
        ws.load(p)
        return ws

    def load(self, p):
        self.k_pool.copy_(p.k_pool)
        self.v_pool.copy_(p.v_pool)
        self.page_table.copy_(p.page_table)
        self.req_pool_indices[:p.batch].copy_(p.req_pool_indices)
        self.seq_lens[:p.batch].copy_(p.seq_lens)
        self.err.zero_()
