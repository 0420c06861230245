"""Seeded random sweeps of the GPU paths against the oracle: shapes, page
sizes, lengths, new-token counts and split counts drawn from a fixed seed, so
that combinations the hand-written cases do not name still get compared
(every case is reproducible from its index).  PKV_RANDOM_CASES=n runs cases
0 .. n-1 of each sweep instead of the default counts."""
import os

import numpy as np
import pytest
import torch

import oracle.ref as R
import pkv_inputs as W
from paged_kv_decode_bind_gb300 import Workspace
from paged_kv_decode_bind_gb300 import _abi as A
from parity import check_attention, run_steps
from test_gpu_extend import KERNS, _indptr, _slots, _compare, run_extend

pytestmark = pytest.mark.gpu
_N = int(os.environ.get("PKV_RANDOM_CASES", "0"))


def _cases(default):
    return range(_N or default)


def _shape(rng, g16_hkv=(1, 2), hkv=(1, 2, 4)):
    G = int(rng.choice([1, 2, 4, 8, 16]))
    Hkv = int(rng.choice(g16_hkv if G == 16 else hkv))
    return G, Hkv, int(rng.choice([64, 128]))


@pytest.mark.parametrize("case", _cases(24))
def test_random_causal_extend(cuda, case):
    # Causal extend, both kernels, 1 / 2 / 7 / 33 splits, page sizes 16 and 32.
    rng = np.random.default_rng(7100 + case)
    G, Hkv, D = _shape(rng, hkv=(1, 2, 4))
    P = int(rng.choice([16, 32]))
    B = int(rng.integers(1, 4))
    lens = [int(rng.integers(1, 600)) for _ in range(B)]
    qo = [int(rng.integers(0, min(L, 70) + 1)) for L in lens]
    if sum(qo) == 0:
        qo[0] = 1
    S = int(rng.choice([1, 2, 7, 33]))
    flags = A.PKV_FLAG_OUT_F32 if rng.integers(0, 2) else 0
    T, Hq = sum(qo), G * Hkv
    rows = sorted({(int(rng.integers(T)), int(rng.integers(Hq))) for _ in range(30)})
    for kern in KERNS:
        got, ref, want, _ = run_extend(cuda, lens=lens, qo=qo, Hq=Hq, Hkv=Hkv, D=D, P=P,
                                       seed=1000 + case, NL=1, layer=0, rows=rows, S=S,
                                       flags=flags | KERNS[kern])
        _compare(got, ref, want, f"case {case} {kern} S={S}")


@pytest.mark.parametrize("case", _cases(16))
def test_random_full_extend(cuda, case):
    # No causal mask (a cascade's prefix pass): every query row of request b
    # attends keys [0, L_b), more rows than keys allowed, empty contexts
    # included; the oracle is decode attention of each row over the context.
    rng = np.random.default_rng(7200 + case)
    G, Hkv, D = _shape(rng, hkv=(1, 2))
    P = int(rng.choice([16, 32]))
    B = int(rng.integers(1, 4))
    lens = [int(rng.integers(0, 600)) for _ in range(B)]
    qo = [int(rng.integers(0, 70)) for _ in range(B)]
    if sum(qo) == 0:
        qo[0] = 1
    S = int(rng.choice([1, 2, 7, 33]))
    Hq, T, mq = G * Hkv, sum(qo), max(qo)
    p = W.make_problem("full", batch=B, n_layers=1, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=D,
                       page_size=P, seq_lens=[max(1, L) for L in lens], seed=2000 + case)
    ws = Workspace.from_problem(p, max_splits=mq * S if S > 1 else 1)
    for b in range(B):
        ws.seq_lens[b] = lens[b]
    q = W.normal_bf16((T, Hq, D), 2100 + case)
    slots, qb = _slots(p), R.tensor_bits(q)
    kb, vb = R.tensor_bits(p.k_pool), R.tensor_bits(p.v_pool)
    ref = np.zeros((T, Hq, D))
    r0 = 0
    for b in range(B):
        if qo[b] and lens[b]:
            ref[r0:r0 + qo[b]], _ = R.decode_attention(qb[r0:r0 + qo[b]], kb, vb, 0,
                                                       [slots[b][:lens[b]]] * qo[b], p.scale, Hkv)
        r0 += qo[b]
    for kern in KERNS:
        ws.err.zero_()
        out = torch.full((T, Hq, D), 7.0, dtype=torch.float32, device=cuda)
        A.pkv_extend_attn(ws, B, 0, _indptr(qo, cuda), mq, q.to(cuda), out, p.scale,
                          num_splits=S,
                          flags=A.PKV_FLAG_EXTEND_FULL | A.PKV_FLAG_OUT_F32 | KERNS[kern])
        torch.cuda.synchronize()
        assert int(ws.err.item()) == 0
        check_attention(out.to(torch.float64).cpu().numpy(), ref, f"case {case} {kern} S={S}")


@pytest.mark.parametrize("case", _cases(24))
def test_random_decode(cuda, case):
    # Steady decode steps, fused and unfused, the tensor-map and the gather
    # producers, page sizes 1 (flat) to 48, batches 1 to 40, 1 to 16 splits.
    rng = np.random.default_rng(7300 + case)
    G, Hkv, D = _shape(rng, hkv=(1, 2, 4))
    P = int(rng.choice([1, 8, 16, 32, 48]))
    B = int(rng.choice([1, 3, 17, 40]))
    lens = [int(rng.integers(1, 900)) for _ in range(B)]
    S = int(rng.choice([1, 2, 5, 16]))
    fused = bool(rng.integers(0, 2))
    flags = A.PKV_FLAG_OUT_F32 if rng.integers(0, 4) == 0 else 0
    if P % 16 == 0 and rng.integers(0, 3) == 0:
        flags |= A.PKV_FLAG_FORCE_GATHER
    p = W.make_problem("random", batch=B, n_layers=2, n_q_heads=G * Hkv, n_kv_heads=Hkv,
                       head_dim=D, page_size=P, seq_lens=lens, steps=2, seed=3000 + case)
    heads = [(int(rng.integers(B)), int(rng.integers(G * Hkv))) for _ in range(24)]
    run_steps(p, S=S, steps=2, heads=heads, flags=flags, fused=fused, check_pool=False)
