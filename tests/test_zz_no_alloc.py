"""pkv_decode_attn_static_scratch: the decode entry point for callers that
cannot allocate device memory (for example a plugin that is handed only its
input and output buffers).  It keeps the split partials in the library's own
static device array, so the caller passes no o_part / ml_part at all.

Checked through the C ABI against the regular pkv_decode_attn +
pkv_merge_partials path on the same inputs, on two calls in a row (with
different split counts, so stale contents left by the first call would show
up in the second), within the attention tolerance the parity tests use.
This file sorts last so a run that stops at the first failure has already
run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import pkv_inputs as W
from paged_kv_decode_bind_gb300 import DecodeRunner, Workspace
from paged_kv_decode_bind_gb300 import _abi as A

from parity import bf16_to_f64, check_attention

pytestmark = pytest.mark.gpu


def _regular(ws, B, layer, q, scale, S):
    A.pkv_decode_attn(ws, B, layer, q, scale, S, 0)
    A.pkv_merge_partials(ws, B, S, 0)
    torch.cuda.synchronize()
    return bf16_to_f64(ws.out_bf16(B)).copy()


def test_static_scratch_matches_regular_path(cuda):
    p = W.workload("gqa4_b4_paged", shrink=8, steps=1)
    B = p.batch
    ws = Workspace.from_problem(p, max_splits=8)
    run = DecodeRunner(ws, B, num_splits=1, scale=p.scale)
    q, k, v = W.step_inputs(p, 0)
    run.q_in.copy_(q)
    run.k_in.copy_(k)
    run.v_in.copy_(v)
    run.bind()
    for layer in range(p.n_layers):
        A.pkv_bind_step(ws, B, A.PKV_BIND_APPEND_ONLY, layer, 1, run.k_in[layer], run.v_in[layer])
    calls = [(0, 6), (1, 3)]  # (layer, num_splits) of the two calls in a row
    ref = [_regular(ws, B, l, run.q_in[l], p.scale, S) for l, S in calls]

    # A copy of the workspace struct with no partial buffers at all.
    bare = A.PkvWorkspace()
    ctypes.pointer(bare)[0] = ws.struct
    bare.o_part = None
    bare.ml_part = None
    got = []
    for l, S in calls:
        A.pkv_decode_attn_static_scratch(bare, B, l, run.q_in[l], p.scale, S, 0)
        torch.cuda.synchronize()
        got.append(bf16_to_f64(ws.out_bf16(B)).copy())
    for (l, S), r, g in zip(calls, ref, got):
        check_attention(g, r, f"static scratch layer {l} S={S}")
    assert int(ws.err.item()) == 0


def test_static_scratch_rejects_oversize(cuda):
    p = W.workload("gqa4_b4_paged", shrink=8, steps=1)
    ws = Workspace.from_problem(p, max_splits=1)
    big = A.PkvWorkspace()
    ctypes.pointer(big)[0] = ws.struct
    big.max_batch = 4096
    big.max_splits = 1 << 20
    q = torch.zeros((4096, p.n_q_heads, p.head_dim), dtype=torch.bfloat16, device="cuda")
    # 4096 * 32 heads * 64 splits * 130 floats * 4 B > 8 MiB
    s = A.pkv_decode_attn_static_scratch(big, 4096, 0, q, p.scale, 64, 0, check=False)
    assert s == A.PKV_ERR_CAPACITY
