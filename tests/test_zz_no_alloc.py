"""pkv_decode_attn_static_scratch: the decode entry point for callers that
cannot allocate device memory (for example a plugin that is handed only its
input and output buffers).  It keeps the split partials in the library's own
static device array, so the caller passes no o_part / ml_part at all.

Checked through the C ABI against the regular pkv_decode_attn +
pkv_merge_partials path on the same inputs and against the CPU oracle, on
two split calls in a row (with different split counts, so stale contents
left by the first call would show up in the second) and then an unsplit
call, for the tensor-core kernel, the CUDA-core kernel and the fp32 output
with lse, within the attention tolerance the parity tests use.  This file
sorts last so a run that stops at the first failure has already run every
other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle.ref as R
import pkv_inputs as W
from paged_kv_decode_bind_gb300 import DecodeRunner, Workspace
from paged_kv_decode_bind_gb300 import _abi as A

from parity import OracleState, bf16_to_f64, check_attention

pytestmark = pytest.mark.gpu

FLAGS = {"mma": 0, "simt": A.PKV_FLAG_FORCE_SIMT,
         "lse_f32": A.PKV_FLAG_WRITE_LSE | A.PKV_FLAG_OUT_F32}
# (layer, num_splits): two split calls in a row, then one unsplit
CALLS = [(0, 6), (1, 3), (1, 1)]


def _out(ws, B, flags):
    if flags & A.PKV_FLAG_OUT_F32:
        return ws.out_f32(B).cpu().numpy().astype(np.float64).copy()
    return bf16_to_f64(ws.out_bf16(B)).copy()


def _regular(ws, B, layer, q, scale, S, flags):
    A.pkv_decode_attn(ws, B, layer, q, scale, S, flags)
    A.pkv_merge_partials(ws, B, S, flags)
    torch.cuda.synchronize()
    return _out(ws, B, flags), ws.lse[:B].cpu().numpy().copy()


@pytest.mark.parametrize("kind", list(FLAGS))
def test_static_scratch_matches_regular_path_and_oracle(cuda, kind):
    flags = FLAGS[kind]
    p = W.workload("gqa4_b4_paged", shrink=8, steps=1)
    B = p.batch
    ws = Workspace.from_problem(p, max_splits=8)
    run = DecodeRunner(ws, B, num_splits=1, scale=p.scale)
    q, k, v = W.step_inputs(p, 0)
    run.q_in.copy_(q)
    run.k_in.copy_(k)
    run.v_in.copy_(v)
    run.bind()
    st = OracleState(p)
    st.bind()
    for layer in range(p.n_layers):
        A.pkv_bind_step(ws, B, A.PKV_BIND_APPEND_ONLY, layer, 1, run.k_in[layer], run.v_in[layer])
        st.append(layer, R.tensor_bits(k)[layer], R.tensor_bits(v)[layer])
    ref = [_regular(ws, B, l, run.q_in[l], p.scale, S, flags) for l, S in CALLS]

    # A copy of the workspace struct with no partial buffers at all.
    bare = A.PkvWorkspace()
    ctypes.pointer(bare)[0] = ws.struct
    bare.o_part = None
    bare.ml_part = None
    got = []
    for l, S in CALLS:
        A.pkv_decode_attn_static_scratch(bare, B, l, run.q_in[l], p.scale, S, flags)
        torch.cuda.synchronize()
        got.append((_out(ws, B, flags), ws.lse[:B].cpu().numpy().copy()))
    qbits = R.tensor_bits(q)
    for (l, S), (r, rl), (g, gl) in zip(CALLS, ref, got):
        what = f"static scratch {kind} layer {l} S={S}"
        check_attention(g, r, what + " vs the regular path")
        o_ref, lse_ref = st.attention(l, qbits[l])
        check_attention(g, o_ref, what + " vs the oracle")
        if flags & A.PKV_FLAG_WRITE_LSE:
            assert np.abs(gl - lse_ref).max() <= 1e-3, what
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
    # a shape that would make the size product non-positive is rejected first
    bad = A.PkvWorkspace()
    ctypes.pointer(bad)[0] = ws.struct
    bad.head_dim = -128
    s = A.pkv_decode_attn_static_scratch(bad, 4, 0, q, p.scale, 64, 0, check=False)
    assert s == A.PKV_ERR_INVALID
