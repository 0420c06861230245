"""libpkv loads, exports every symbol include/pkv.h declares, and rejects bad
arguments on the host (no GPU needed: every call here fails validation or is
host-only, so nothing is launched)."""
import ctypes
import os
import re

import pytest

import paged_kv_decode_bind_gb300 as P
from paged_kv_decode_bind_gb300 import _abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")


def _declared():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_0-9]+)\s*\(", text)))


def test_exports_match_header():
    lib = _abi.load()
    declared = _declared()
    assert declared, "no declarations parsed"
    assert sorted(_abi.EXPORTS) == declared
    for name in declared:
        assert hasattr(lib, name), name


def test_struct_layout():
    # 12 int32 shape fields, 16 pointers, then max_seq_len (and 4 bytes of
    # tail padding to the pointers' 8-byte alignment) on LP64.
    assert ctypes.sizeof(_abi.PkvWorkspace) == 12 * 4 + 16 * 8 + 8
    assert _abi.PkvWorkspace.k_pool.offset == 48
    assert _abi.PkvWorkspace.max_seq_len.offset == 12 * 4 + 16 * 8


def _ws(**kw):
    shape = dict(n_layers=2, pool_slots=64, n_q_heads=8, n_kv_heads=2, head_dim=128,
                 page_size=16, index_mode=0, max_batch=4, max_reqs=8, max_pages_per_req=4,
                 max_splits=4, max_total_tokens=0, max_seq_len=0)
    fake = 1 << 20  # non-null, 16-byte aligned; never dereferenced (validation fails first)
    ptrs = dict(k_pool=fake, v_pool=fake, req_pool_indices=fake, page_table=fake,
                seq_lens=fake, position_ids=fake, kv_indptr=fake, out_loc=fake,
                kv_indices=fake, o_part=fake, ml_part=fake, out=fake, lse=fake, err=fake,
                split_counters=fake, work_plan=fake)
    shape.update({k: v for k, v in kw.items() if k in shape})
    ptrs.update({k: v for k, v in kw.items() if k in ptrs})
    return _abi.PkvWorkspace(**shape, **ptrs)


def test_workspace_bytes():
    ws = _ws()
    assert P.pkv_workspace_bytes(ws, "k_pool") == 2 * 64 * 2 * 128 * 2
    assert P.pkv_workspace_bytes(ws, "o_part") == 4 * 8 * 4 * 128 * 4
    assert P.pkv_workspace_bytes(ws, "ml_part") == 4 * 8 * 4 * 2 * 4
    assert P.pkv_workspace_bytes(ws, "kv_indptr") == 5 * 4
    assert P.pkv_workspace_bytes(ws, "page_table") == 8 * 4 * 4
    assert P.pkv_workspace_bytes(ws, "out") == 4 * 8 * 128 * 4
    assert P.pkv_workspace_bytes(ws, "nope") == 0


@pytest.mark.parametrize("kw,batch,layer,splits,flags,status", [
    (dict(head_dim=96), 1, 0, 1, 0, P.PKV_ERR_UNSUPPORTED),
    (dict(n_q_heads=24, n_kv_heads=2), 1, 0, 1, 0, P.PKV_ERR_UNSUPPORTED),   # G = 12
    (dict(n_q_heads=7), 1, 0, 1, 0, P.PKV_ERR_INVALID),                      # Hq % Hkv
    (dict(), 5, 0, 1, 0, P.PKV_ERR_CAPACITY),                                # batch > max
    (dict(), 1, 2, 1, 0, P.PKV_ERR_CAPACITY),                                # layer >= NL
    (dict(), 1, 0, 5, 0, P.PKV_ERR_CAPACITY),                                # splits > max
    (dict(), 1, 0, 0, 0, P.PKV_ERR_INVALID),                                 # splits < 1
    (dict(err=None), 1, 0, 1, 0, P.PKV_ERR_INVALID),
    (dict(k_pool=(1 << 20) + 8), 1, 0, 1, 0, P.PKV_ERR_INVALID),             # misaligned
    (dict(o_part=None), 1, 0, 2, 0, P.PKV_ERR_INVALID),
    (dict(o_part=(1 << 20) + 8), 1, 0, 2, 0, P.PKV_ERR_INVALID),            # misaligned
    (dict(ml_part=(1 << 20) + 4), 1, 0, 2, 0, P.PKV_ERR_INVALID),           # (m, l) pairs
    (dict(lse=None), 1, 0, 1, P.PKV_FLAG_WRITE_LSE, P.PKV_ERR_INVALID),
    (dict(index_mode=1), 1, 0, 1, 0, P.PKV_ERR_INVALID),                     # flat needs P == 1
    (dict(pool_slots=60), 1, 0, 1, 0, P.PKV_ERR_INVALID),                    # slots % P
    (dict(max_seq_len=-1), 1, 0, 1, 0, P.PKV_ERR_INVALID),
    (dict(n_q_heads=32, n_kv_heads=2), 1, 0, 1, P.PKV_FLAG_FORCE_SIMT, P.PKV_ERR_UNSUPPORTED),
    (dict(), 1, 0, 1, P.PKV_FLAG_FORCE_SIMT | P.PKV_FLAG_FORCE_MMA, P.PKV_ERR_INVALID),
    (dict(), 1, 0, 1, P.PKV_FLAG_FORCE_SIMT | P.PKV_FLAG_FORCE_GATHER, P.PKV_ERR_INVALID),
    (dict(n_q_heads=64, n_kv_heads=2), 1, 0, 1, P.PKV_FLAG_FORCE_MMA, P.PKV_ERR_UNSUPPORTED),
])
def test_decode_host_validation(kw, batch, layer, splits, flags, status):
    # Every case here must fail host validation: nothing may be launched.
    ws = _ws(**kw)
    got = P.pkv_decode_attn(ws, batch, layer, 1 << 20, 0.1, splits, flags, 0, check=False)
    assert got == status, (got, status)


def test_bind_and_merge_host_validation():
    ws = _ws()
    assert P.pkv_bind_step(ws, 1, 7, 0, 0, None, None, 0, check=False) == P.PKV_ERR_INVALID
    assert P.pkv_bind_step(ws, 9, 0, 0, 0, None, None, 0, check=False) == P.PKV_ERR_CAPACITY
    assert P.pkv_bind_step(ws, 1, 2, 1, 2, 1 << 20, 1 << 20, 0, check=False) == \
        P.PKV_ERR_CAPACITY
    assert P.pkv_bind_step(ws, 1, 2, 0, 1, None, None, 0, check=False) == P.PKV_ERR_INVALID
    assert P.pkv_bind_step(_ws(seq_lens=None), 1, 0, 0, 0, None, None, 0, check=False) == \
        P.PKV_ERR_INVALID
    # batch 0 and one split are valid no-ops that launch nothing
    assert P.pkv_bind_step(ws, 0, 0, 0, 0, None, None, 0, check=False) == P.PKV_OK
    assert P.pkv_merge_partials(ws, 2, 1, 0, 0, check=False) == P.PKV_OK
    assert P.pkv_merge_partials(ws, 2, 9, 0, 0, check=False) == P.PKV_ERR_CAPACITY
    assert P.pkv_decode_attn(ws, 0, 0, 1 << 20, 0.1, 1, 0, 0, check=False) == P.PKV_OK
    assert P.pkv_merge_partials(None, 1, 2, 0, 0, check=False) == P.PKV_ERR_INVALID
    assert P.pkv_merge_partials(_ws(ml_part=(1 << 20) + 4), 1, 2, 0, 0, check=False) == \
        P.PKV_ERR_INVALID
    # fused layer: k/v rows both or neither; split counters needed when S > 1
    f = 1 << 20
    assert P.pkv_decode_layer(ws, 1, 0, f, f, None, 0.1, 1, 0, 0, check=False) == \
        P.PKV_ERR_INVALID
    assert P.pkv_decode_layer(_ws(split_counters=None), 1, 0, f, f, f, 0.1, 2, 0, 0,
                              check=False) == P.PKV_ERR_INVALID
    assert P.pkv_decode_layer(ws, 5, 0, f, f, f, 0.1, 1, 0, 0, check=False) == \
        P.PKV_ERR_CAPACITY
    assert P.pkv_decode_layer(ws, 0, 0, f, f, f, 0.1, 2, 0, 0, check=False) == P.PKV_OK


def test_extend_host_validation():
    # Every case fails (or no-ops) on the host: nothing is launched.
    f = 1 << 20
    X = P.pkv_extend_attn
    cases = [
        (dict(n_q_heads=24, n_kv_heads=2), 1, 0, f, 4, f, f, 0, P.PKV_ERR_UNSUPPORTED),  # G = 12
        (dict(head_dim=96), 1, 0, f, 4, f, f, 0, P.PKV_ERR_UNSUPPORTED),
        (dict(), 5, 0, f, 4, f, f, 0, P.PKV_ERR_CAPACITY),                           # batch
        (dict(), 1, 2, f, 4, f, f, 0, P.PKV_ERR_CAPACITY),                           # layer
        (dict(), 1, 0, None, 4, f, f, 0, P.PKV_ERR_INVALID),                         # qo_indptr
        (dict(), 1, 0, f, 4, None, f, 0, P.PKV_ERR_INVALID),                         # q
        (dict(), 1, 0, f, 4, f + 8, f, 0, P.PKV_ERR_INVALID),                        # misaligned
        (dict(), 1, 0, f, -1, f, f, 0, P.PKV_ERR_INVALID),                           # max_qo_len
        (dict(), 1, 0, f, 4, f, f, P.PKV_FLAG_FORCE_SIMT, P.PKV_ERR_INVALID),        # flag
        (dict(lse=None), 1, 0, f, 4, f, f, P.PKV_FLAG_WRITE_LSE, P.PKV_ERR_INVALID),
        (dict(), 2, 0, f, 4, f, f, P.PKV_FLAG_WRITE_LSE, P.PKV_ERR_CAPACITY),        # 8 rows
        (dict(), 0, 0, f, 4, f, f, 0, P.PKV_OK),                                     # no batch
        (dict(), 1, 0, f, 0, f, f, 0, P.PKV_OK),                                     # no tokens
        (dict(), 0, 0, f, 4, f, f, P.PKV_FLAG_PLAN_EARLY, P.PKV_OK),                 # accepted
    ]
    for kw, batch, layer, qo, mq, q, out, flags, status in cases:
        got = X(_ws(**kw), batch, layer, qo, mq, q, out, 0.1, num_splits=1, flags=flags,
                stream=0, check=False)
        assert got == status, (kw, batch, layer, mq, flags, got, status)
    # splits: partials need o_part / ml_part with room for batch * max_qo_len * S rows
    assert X(_ws(), 1, 0, f, 4, f, f, 0.1, num_splits=0, stream=0, check=False) == \
        P.PKV_ERR_INVALID
    assert X(_ws(o_part=None), 1, 0, f, 4, f, f, 0.1, num_splits=2, stream=0, check=False) == \
        P.PKV_ERR_INVALID
    assert X(_ws(ml_part=f + 4), 1, 0, f, 4, f, f, 0.1, num_splits=2, stream=0, check=False) == \
        P.PKV_ERR_INVALID
    assert X(_ws(), 4, 0, f, 4, f, f, 0.1, num_splits=2, stream=0, check=False) == \
        P.PKV_ERR_CAPACITY  # 4 * 4 * 2 rows > max_batch 4 * max_splits 4
    A = P.pkv_extend_append
    assert A(_ws(), 1, 0, f, 4, f, None, 0, check=False) == P.PKV_ERR_INVALID
    assert A(_ws(), 5, 0, f, 4, f, f, 0, check=False) == P.PKV_ERR_CAPACITY
    assert A(_ws(), 1, 0, f, 0, f, f, 0, check=False) == P.PKV_OK


def test_merge_lse_host_validation():
    f = 1 << 20
    M = P.pkv_merge_lse
    assert M(-1, 128, f, f, f, f, f, None, 0, 0, check=False) == P.PKV_ERR_INVALID
    assert M(4, 96, f, f, f, f, f, None, 0, 0, check=False) == P.PKV_ERR_UNSUPPORTED
    assert M(4, 128, None, f, f, f, f, None, 0, 0, check=False) == P.PKV_ERR_INVALID
    assert M(4, 128, f + 8, f, f, f, f, None, 0, 0, check=False) == P.PKV_ERR_INVALID
    assert M(4, 128, f, f, f, f, f, None, P.PKV_FLAG_WRITE_LSE, 0, check=False) == \
        P.PKV_ERR_INVALID
    assert M(0, 128, f, f, f, f, f, None, 0, 0, check=False) == P.PKV_OK


def test_choose_splits():
    ws = _ws(max_splits=128, n_kv_heads=8, n_q_heads=32)
    # one 65536-token request: 38 splits x 8 heads = 304 units, one per
    # resident block of 152 SMs x 2
    assert P.pkv_choose_splits(ws, 1, 65536, 65536, 152) == 38
    # four such requests: 19 splits -> 608 units = exactly two waves
    assert P.pkv_choose_splits(ws, 4, 65600, 4 * 65568, 152) == 19
    # mixed lengths: fluid share plus half a wave decides
    assert P.pkv_choose_splits(ws, 4, 2048, 6500, 152) == 12
    assert P.pkv_choose_splits(ws, 16, 8192, 14500, 152) == 37
    # no total given: batch * max, treated as uniform
    assert P.pkv_choose_splits(ws, 4, 2048, 0, 152) == 9
    assert P.pkv_choose_splits(_ws(max_splits=4), 1, 65536, 65536, 152) == 4
    assert P.pkv_choose_splits(ws, 0, 10, 10, 152) == 1


def test_choose_pieces():
    ws = _ws(max_splits=128, n_kv_heads=8, n_q_heads=32)
    # share = ceil(8 * 65536 / 304) = 1725 -> 3 + 65535 // 1725
    assert P.pkv_choose_pieces(ws, 1, 65536, 65536, 152) == 40
    # share = ceil(8 * 262272 / 304) = 6902 -> 3 + 65599 // 6902
    assert P.pkv_choose_pieces(ws, 4, 65600, 4 * 65568, 152) == 12
    # skewed: share = ceil(8 * 14500 / 304) = 382 -> 3 + 8191 // 382
    assert P.pkv_choose_pieces(ws, 16, 8192, 14500, 152) == 24
    # share = ceil(8 * 6500 / 304) = 172 -> 3 + 2047 // 172
    assert P.pkv_choose_pieces(ws, 4, 2048, 6500, 152) == 14
    # the share floor of 128 tokens
    assert P.pkv_choose_pieces(ws, 1, 300, 300, 152) == 5
    # four tiles or fewer: no split
    assert P.pkv_choose_pieces(ws, 1, 256, 256, 152) == 1
    assert P.pkv_choose_pieces(ws, 64, 192, 64 * 192, 152) == 1
    assert P.pkv_choose_pieces(_ws(max_splits=4), 1, 65536, 65536, 152) == 4
    assert P.pkv_choose_pieces(_ws(max_splits=1), 1, 65536, 65536, 152) == 1
    assert P.pkv_choose_pieces(ws, 0, 10, 10, 152) == 1


def test_steady_predicate_matches_oracle():
    import oracle.ref as R
    cases = [([4, 9], [10, 3], [4, 9], [11, 4]), ([4, 9], [10, 3], [9, 4], [4, 11]),
             ([4, 9], [10, 3], [4, 9], [11, 5]), ([1], [0], [1, 2], [1, 1]),
             (None, None, [1], [1]), ([7], [1], [7], [2])]
    for c in cases:
        assert P.pkv_is_steady_increment(*c) == R.is_steady_increment(*c), c


def test_status_strings():
    for s in range(5):
        assert P.pkv_status_string(s)
    assert "sm_103a" in P.pkv_version()


def test_bind_tracker_sequence():
    # The host record of the last bind: the first step and any step whose task
    # set or lengths did not just grow by one token rebuild; the record moves
    # to every step it was asked about, steady or not.
    t = P.BindTracker()
    S, RB = P.PKV_BIND_STEADY, P.PKV_BIND_REBUILD
    assert t.mode([7, 3], [10, 4]) == RB          # nothing bound yet
    assert t.mode([7, 3], [11, 5]) == S
    assert t.mode([7, 3], [12, 6]) == S
    assert t.mode([7, 3], [14, 7]) == RB          # one request grew by two
    assert t.mode([7, 3], [15, 8]) == S           # ... against the rebuilt record
    assert t.mode([3, 7], [9, 16]) == RB          # same tasks, other order
    assert t.mode([3, 7, 5], [10, 17, 1]) == RB   # a task joined
    assert t.mode([3, 7, 5], [11, 18, 2]) == S
    assert t.mode([], []) == RB                   # an empty batch is never steady


def test_choose_extend_splits():
    # Fill the resident blocks, no split under 256 keys, within the partials'
    # room.  Page sizes that are a multiple of 16 take the tcgen05 kernel:
    # 128 query rows per CTA, one CTA per SM at D = 128.
    big = _ws(n_q_heads=32, n_kv_heads=8, max_batch=64, max_splits=4096)
    C = P.pkv_choose_extend_splits
    # 64 new tokens at G = 4: 2 blocks per head, 8 heads, one request: 16 units
    assert C(big, 1, 64, 32832, 152) == 9
    assert C(big, 4, 256, 900, 152) == 1           # 256 units already fill the SMs
    assert C(big, 1, 64, 600, 152) == 2            # 600 keys: two splits of >= 256
    assert C(big, 1, 64, 100, 152) == 1
    # the partials' room: max_batch * max_splits rows over batch * max_qo_len
    assert C(_ws(n_q_heads=32, n_kv_heads=8, max_batch=4, max_splits=4), 1, 4, 32832, 152) == 4
    assert C(None, 1, 64, 32832, 152) == 1
    assert C(big, 0, 64, 32832, 152) == 1
    assert C(big, 1, 64, 32832, 0) == 1
    ws = lambda Hq, Hkv, **kw: _ws(n_q_heads=Hq, n_kv_heads=Hkv, max_batch=64, max_splits=4096,
                                   **kw)
    # G = 8: 16 tokens per CTA, 3 x 2 x 2 = 12 units, 152 / 12 = 12, 3000 keys allow 11
    assert C(ws(16, 2), 2, 40, 3000, 152) == 11
    # G = 1: 128 tokens per CTA, 24 units, 6 by the SMs, 700 keys allow 2
    assert C(ws(8, 8), 3, 17, 700, 152) == 2
    # G = 16: 8 tokens per CTA, 2 units: 76 splits
    assert C(ws(32, 2), 1, 1, 70000, 152) == 76
    # head_dim 64: the same geometry
    assert C(ws(32, 2, head_dim=64), 1, 1, 70000, 152) == 76
    # page size 8: the warp-level kernel, 64 rows per block (4 tokens at
    # G = 16), two blocks per SM
    assert C(ws(32, 2, page_size=8), 1, 1, 70000, 152) == 152



def test_static_scratch_host_validation():
    # Rejected before any CUDA call: a shape that would make the scratch size
    # product non-positive, and a size beyond the static array.
    q = 1 << 20
    assert P.pkv_decode_attn_static_scratch(_ws(head_dim=-128), 1, 0, q, 0.1, 4, 0,
                                            check=False) == P.PKV_ERR_INVALID
    assert P.pkv_decode_attn_static_scratch(_ws(n_q_heads=0), 1, 0, q, 0.1, 4, 0,
                                            check=False) == P.PKV_ERR_INVALID
    big = _ws(max_batch=4096)
    assert P.pkv_decode_attn_static_scratch(big, 4096, 0, q, 0.1, 64, 0,
                                            check=False) == P.PKV_ERR_CAPACITY
