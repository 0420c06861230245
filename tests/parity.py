"""Shared driver for the GPU parity tests: runs one or more steady decode
steps through libpkv and through the CPU oracle on the same seeded inputs
and compares them.

Tolerances (attention output, bf16 in / fp32 accumulate vs fp64):
  max |gpu - ref| <= 1e-2  and  max |gpu - ref| / max |ref| <= 2e-2
Cross-split agreement (fp32 outputs): max |a - b| <= 1e-3.
Split partials vs the oracle's: |o| 1e-3 abs, m 1e-3 abs, l 1e-4 rel.
Metadata, kv_indices and appended pool rows: bit-exact.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle.ref as R
import pkv_inputs as W
from paged_kv_decode_bind_gb300 import DecodeRunner, Workspace
from paged_kv_decode_bind_gb300 import _abi as A

ATOL = 1e-2
NRTOL = 2e-2
SPLIT_ATOL = 1e-3


def bf16_to_f64(t):
    return t.detach().to("cpu").to(torch.float64).numpy()


def check_attention(got, ref, what=""):
    err = np.abs(got - ref)
    mx = float(err.max()) if err.size else 0.0
    scale = float(np.abs(ref).max()) if ref.size else 0.0
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert mx <= ATOL, f"{what}: max abs err {mx:.3e} > {ATOL}"
    if scale > 0:
        assert mx / scale <= NRTOL, f"{what}: normwise rel err {mx / scale:.3e} > {NRTOL}"
    return mx


class OracleState:
    """Oracle-side copy of the pools and metadata, advanced step by step."""

    def __init__(self, p: W.DecodeProblem):
        self.p = p
        self.kb = R.tensor_bits(p.k_pool).copy()
        self.vb = R.tensor_bits(p.v_pool).copy()
        self.lens = p.seq_lens.tolist()
        self.table = p.page_table.numpy()
        self.rows = p.req_pool_indices.numpy()
        self.meta = None

    def bind(self, mode=R.STEADY):
        self.meta = R.bind(self.lens, req_pool_indices=self.rows, page_table=self.table,
                           page_size=self.p.page_size, mode=mode,
                           index_mode=R.FLAT if self.p.index_mode == 1 else R.PAGE_TABLE)
        self.lens = self.meta["seq_lens"]
        return self.meta

    def append(self, layer, k_bits, v_bits):
        for b, loc in enumerate(self.meta["out_loc"]):
            self.kb[layer, loc] = k_bits[b]
            self.vb[layer, loc] = v_bits[b]

    def slots(self):
        p = self.p
        if p.index_mode == 1:
            return [R.token_slots(b, self.lens[b], index_mode=R.FLAT,
                                  kv_indptr=self.meta["kv_indptr"],
                                  kv_indices=self.meta["kv_indices"]) for b in range(p.batch)]
        return [R.token_slots(b, self.lens[b], page_table=self.table, req_pool_indices=self.rows,
                              page_size=p.page_size) for b in range(p.batch)]

    def attention(self, layer, q_bits, heads=None):
        return R.decode_attention(q_bits, self.kb, self.vb, layer, self.slots(), self.p.scale,
                                  self.p.n_kv_heads, heads=heads)

    def partials(self, layer, q_bits, S, heads=None):
        return R.split_partials(q_bits, self.kb, self.vb, layer, self.slots(), self.p.scale,
                                self.p.n_kv_heads, S, self.p.page_size, self.lens, heads=heads)


def check_meta(ws, st: OracleState, B):
    m = st.meta
    assert ws.seq_lens[:B].tolist() == m["seq_lens"]
    assert ws.position_ids[:B].tolist() == m["position_ids"]
    assert ws.kv_indptr[:B + 1].tolist() == m["kv_indptr"]
    assert ws.out_loc[:B].tolist() == m["out_loc"]
    if "kv_indices" in m:
        n = len(m["kv_indices"])
        assert ws.kv_indices[:n].tolist() == m["kv_indices"]


def run_steps(p: W.DecodeProblem, *, S=1, steps=1, check_layers=None, heads=None,
              check_partials=False, check_pool=False, flags=0, device="cuda", fused=False,
              plan=False):
    """Run `steps` steady steps; on the last one compare every checked layer.
    plan=True: the fused layers take the step's split plan (pkv_plan_step).
    Returns dict of max errors."""
    ws = Workspace.from_problem(p, max_splits=S, device=device)
    run = DecodeRunner(ws, p.batch, num_splits=S, flags=flags, scale=p.scale, fused=fused,
                       plan=plan)
    assert run.use_plan == (plan and fused and not flags & A.PKV_FLAG_FORCE_SIMT)
    st = OracleState(p)
    B = p.batch
    check_layers = list(range(p.n_layers)) if check_layers is None else check_layers
    out = {"max_err": 0.0}
    for step in range(steps):
        q, k, v = W.step_inputs(p, step)
        run.q_in.copy_(q)
        run.k_in.copy_(k)
        run.v_in.copy_(v)
        run.bind(A.PKV_BIND_STEADY)
        st.bind(R.STEADY)
        kbits, vbits, qbits = R.tensor_bits(k), R.tensor_bits(v), R.tensor_bits(q)
        last = step == steps - 1
        for l in range(p.n_layers):
            run.layer(l)
            st.append(l, kbits[l], vbits[l])
            if not (last and l in check_layers):
                continue
            torch.cuda.synchronize()
            if flags & A.PKV_FLAG_OUT_F32:
                got = ws.out_f32(B).cpu().numpy().astype(np.float64)
            else:
                got = bf16_to_f64(ws.out_bf16(B))
            ref, _ = st.attention(l, qbits[l], heads=heads)
            if heads is not None:
                idx = tuple(np.array(heads).T)
                got, ref = got[idx], ref[idx]
            out["max_err"] = max(out["max_err"],
                                 check_attention(got, ref, f"{p.name} S={S} layer {l}"))
            if check_partials and S > 1 and not fused:
                op_ref, ml_ref = st.partials(l, qbits[l], S, heads=heads)
                n = B * p.n_q_heads * S
                op = ws.o_part.reshape(-1)[:n * p.head_dim].view(B, p.n_q_heads, S, p.head_dim)
                ml = ws.ml_part.reshape(-1)[:n * 2].view(B, p.n_q_heads, S, 2)
                op, ml = op.cpu().numpy().astype(np.float64), ml.cpu().numpy().astype(np.float64)
                if heads is not None:
                    op, op_ref, ml, ml_ref = op[idx], op_ref[idx], ml[idx], ml_ref[idx]
                # splits past a request's end are not written: compare s < n_b
                chunk = R.split_chunk(st.lens, S, p.page_size)
                nb = np.array([-(-L // chunk) for L in st.lens])
                b_idx = np.array(heads)[:, 0] if heads is not None else \
                    np.repeat(np.arange(B), p.n_q_heads).reshape(B, p.n_q_heads)
                live = np.arange(S) < nb[b_idx][..., None]
                assert np.all(ml_ref[..., 1][~live] == 0), "oracle wrote past n_b"
                assert np.all(ml_ref[..., 1][live] > 0)
                assert np.all(ml[..., 1][live] > 0), "a live split came back empty"
                assert np.abs(op[live] - op_ref[live]).max() <= SPLIT_ATOL
                assert np.abs(ml[..., 0][live] - ml_ref[..., 0][live]).max() <= 1e-3
                rel = np.abs(ml[..., 1][live] / ml_ref[..., 1][live] - 1).max()
                assert rel <= 1e-4, rel
        torch.cuda.synchronize()
        check_meta(ws, st, B)
        assert int(ws.err.item()) == 0, f"device error bits {int(ws.err.item())}"
        if fused:
            assert int(ws.split_counters.abs().sum().item()) == 0, "split counters not reset"
    if check_pool:
        assert np.array_equal(R.tensor_bits(ws.k_pool.cpu()), st.kb)
        assert np.array_equal(R.tensor_bits(ws.v_pool.cpu()), st.vb)
    else:
        # appended rows of the last step, every layer
        locs = torch.tensor(st.meta["out_loc"], dtype=torch.long)
        gk = R.tensor_bits(ws.k_pool[:, locs.to(ws.device)].cpu())
        gv = R.tensor_bits(ws.v_pool[:, locs.to(ws.device)].cpu())
        assert np.array_equal(gk, st.kb[:, locs.numpy()])
        assert np.array_equal(gv, st.vb[:, locs.numpy()])
    out["ws"] = ws
    out["runner"] = run
    return out
