"""ctypes binding of libpkv (include/pkv.h): argument marshalling only.

Every function here has the C entry point's name and arguments; tensors are
passed as their device pointers, streams as their CUDA handles.  A missing
library is an error: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkv.so")

PKV_OK, PKV_ERR_INVALID, PKV_ERR_UNSUPPORTED, PKV_ERR_CAPACITY, PKV_ERR_CUDA = range(5)
PKV_BIND_STEADY, PKV_BIND_REBUILD, PKV_BIND_APPEND_ONLY = 0, 1, 2
PKV_IDX_PAGE_TABLE, PKV_IDX_FLAT = 0, 1
PKV_FLAG_OUT_F32, PKV_FLAG_WRITE_LSE, PKV_FLAG_FORCE_SIMT, PKV_FLAG_FORCE_MMA = 1, 2, 4, 8
PKV_FLAG_FORCE_GATHER, PKV_FLAG_PLAN_EARLY, PKV_FLAG_FIXED_CHUNK = 16, 32, 64
PKV_FLAG_USE_PLAN = 128
PKV_FLAG_TEST_SKIP_FIRST_TILE = 256
PKV_FLAG_EXTEND_FULL = 512
PKV_FLAG_EXTEND_WARP_MMA = 1024
PKV_DEVERR_PAGE, PKV_DEVERR_LEN, PKV_DEVERR_TOTAL, PKV_DEVERR_SLOT, PKV_DEVERR_TIMEOUT = \
    1, 2, 4, 8, 16

# Every symbol include/pkv.h declares (checked by the ABI test).
EXPORTS = ("pkv_workspace_bytes", "pkv_bind_step", "pkv_choose_splits", "pkv_choose_pieces",
           "pkv_choose_extend_splits",
           "pkv_decode_attn",
           "pkv_merge_partials", "pkv_decode_layer", "pkv_plan_step",
           "pkv_decode_attn_static_scratch",
           "pkv_extend_attn", "pkv_extend_append", "pkv_merge_lse",
           "pkv_is_steady_increment",
           "pkv_status_string", "pkv_version")
PKV_STATIC_SCRATCH_BYTES = 8 << 20


class PkvWorkspace(ctypes.Structure):
    """Mirror of ``pkv_workspace`` (same field order and types)."""

    _fields_ = [
        ("n_layers", ctypes.c_int32), ("pool_slots", ctypes.c_int32),
        ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
        ("index_mode", ctypes.c_int32), ("max_batch", ctypes.c_int32),
        ("max_reqs", ctypes.c_int32), ("max_pages_per_req", ctypes.c_int32),
        ("max_splits", ctypes.c_int32), ("max_total_tokens", ctypes.c_int32),
        ("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
        ("req_pool_indices", ctypes.c_void_p), ("page_table", ctypes.c_void_p),
        ("seq_lens", ctypes.c_void_p), ("position_ids", ctypes.c_void_p),
        ("kv_indptr", ctypes.c_void_p), ("out_loc", ctypes.c_void_p),
        ("kv_indices", ctypes.c_void_p), ("o_part", ctypes.c_void_p),
        ("ml_part", ctypes.c_void_p), ("out", ctypes.c_void_p),
        ("lse", ctypes.c_void_p), ("err", ctypes.c_void_p),
        ("split_counters", ctypes.c_void_p), ("work_plan", ctypes.c_void_p),
        ("max_seq_len", ctypes.c_int32),
    ]


class PkvError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn}: {status_string(status)} (status {status})")


_lib = None


def load(path: str = LIB_PATH):
    """Load libpkv.so once; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libpkv.so not built at {path}; run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    W = ctypes.POINTER(PkvWorkspace)
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.pkv_workspace_bytes.argtypes = [W, ctypes.c_char_p]
    lib.pkv_workspace_bytes.restype = ctypes.c_size_t
    lib.pkv_bind_step.argtypes = [W, i32, i32, i32, i32, vp, vp, vp]
    lib.pkv_bind_step.restype = i32
    lib.pkv_choose_splits.argtypes = [W, i32, i32, ctypes.c_longlong, i32]
    lib.pkv_choose_splits.restype = i32
    lib.pkv_choose_pieces.argtypes = [W, i32, i32, ctypes.c_longlong, i32]
    lib.pkv_choose_pieces.restype = i32
    lib.pkv_choose_extend_splits.argtypes = [W, i32, i32, i32, i32]
    lib.pkv_choose_extend_splits.restype = i32
    lib.pkv_decode_attn.argtypes = [W, i32, i32, vp, f32, i32, i32, vp]
    lib.pkv_decode_attn.restype = i32
    lib.pkv_merge_partials.argtypes = [W, i32, i32, i32, vp]
    lib.pkv_merge_partials.restype = i32
    lib.pkv_decode_layer.argtypes = [W, i32, i32, vp, vp, vp, f32, i32, i32, vp]
    lib.pkv_decode_layer.restype = i32
    lib.pkv_plan_step.argtypes = [W, i32, i32, i32, vp]
    lib.pkv_plan_step.restype = i32
    lib.pkv_decode_attn_static_scratch.argtypes = [W, i32, i32, vp, f32, i32, i32, vp]
    lib.pkv_decode_attn_static_scratch.restype = i32
    lib.pkv_extend_attn.argtypes = [W, i32, i32, vp, i32, vp, vp, f32, i32, i32, vp]
    lib.pkv_extend_attn.restype = i32
    lib.pkv_extend_append.argtypes = [W, i32, i32, vp, i32, vp, vp, vp]
    lib.pkv_extend_append.restype = i32
    lib.pkv_merge_lse.argtypes = [i32, i32, vp, vp, vp, vp, vp, vp, i32, vp]
    lib.pkv_merge_lse.restype = i32
    p64, p32 = ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int32)
    lib.pkv_is_steady_increment.argtypes = [p64, p32, i32, p64, p32, i32]
    lib.pkv_is_steady_increment.restype = i32
    lib.pkv_status_string.argtypes = [i32]
    lib.pkv_status_string.restype = ctypes.c_char_p
    lib.pkv_version.argtypes = []
    lib.pkv_version.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _ws(ws):
    if ws is None:
        return None
    st = ws.struct if hasattr(ws, "struct") else ws
    return ctypes.byref(st)


def _check(fn, status):
    if status != PKV_OK:
        raise PkvError(fn, status)
    return status


def status_string(status: int) -> str:
    return load().pkv_status_string(int(status)).decode()


def pkv_status_string(status: int) -> str:
    return status_string(status)


def pkv_version() -> str:
    return load().pkv_version().decode()


def pkv_workspace_bytes(ws, which: str) -> int:
    return int(load().pkv_workspace_bytes(_ws(ws), which.encode()))


def pkv_bind_step(ws, batch, mode, layer_begin=0, layer_count=0, k_new=None, v_new=None,
                  stream=None, check=True):
    s = load().pkv_bind_step(_ws(ws), int(batch), int(mode), int(layer_begin), int(layer_count),
                             _ptr(k_new), _ptr(v_new), _stream(stream))
    return _check("pkv_bind_step", s) if check else s


def pkv_choose_splits(ws, batch, max_seq_len_hint, total_tokens_hint, num_sms) -> int:
    return int(load().pkv_choose_splits(_ws(ws), int(batch), int(max_seq_len_hint),
                                        int(total_tokens_hint), int(num_sms)))


def pkv_choose_pieces(ws, batch, max_seq_len_hint, total_tokens_hint, num_sms) -> int:
    return int(load().pkv_choose_pieces(_ws(ws), int(batch), int(max_seq_len_hint),
                                        int(total_tokens_hint), int(num_sms)))


def pkv_choose_extend_splits(ws, batch, max_qo_len, min_seq_len_hint, num_sms) -> int:
    return int(load().pkv_choose_extend_splits(_ws(ws), int(batch), int(max_qo_len),
                                               int(min_seq_len_hint), int(num_sms)))


def pkv_decode_attn(ws, batch, layer, q, scale, num_splits=1, flags=0, stream=None, check=True):
    s = load().pkv_decode_attn(_ws(ws), int(batch), int(layer), _ptr(q), float(scale),
                               int(num_splits), int(flags), _stream(stream))
    return _check("pkv_decode_attn", s) if check else s


def pkv_merge_partials(ws, batch, num_splits, flags=0, stream=None, check=True):
    s = load().pkv_merge_partials(_ws(ws), int(batch), int(num_splits), int(flags),
                                  _stream(stream))
    return _check("pkv_merge_partials", s) if check else s


def pkv_decode_layer(ws, batch, layer, q, k_new, v_new, scale, num_splits=1, flags=0,
                     stream=None, check=True):
    s = load().pkv_decode_layer(_ws(ws), int(batch), int(layer), _ptr(q), _ptr(k_new),
                                _ptr(v_new), float(scale), int(num_splits), int(flags),
                                _stream(stream))
    return _check("pkv_decode_layer", s) if check else s


def pkv_plan_step(ws, batch, num_splits=1, flags=0, stream=None, check=True):
    s = load().pkv_plan_step(_ws(ws), int(batch), int(num_splits), int(flags), _stream(stream))
    return _check("pkv_plan_step", s) if check else s


def pkv_decode_attn_static_scratch(ws, batch, layer, q, scale, num_splits=1, flags=0,
                                   stream=None, check=True):
    """Decode attention + merge with the partials in the library's static
    device array (for callers that cannot allocate device memory)."""
    s = load().pkv_decode_attn_static_scratch(_ws(ws), int(batch), int(layer), _ptr(q),
                                              float(scale), int(num_splits), int(flags),
                                              _stream(stream))
    return _check("pkv_decode_attn_static_scratch", s) if check else s


def pkv_extend_attn(ws, batch, layer, qo_indptr, max_qo_len, q, out, scale, num_splits=1,
                    flags=0, stream=None, check=True):
    """Causal extend attention of each request's newest tokens (device
    qo_indptr int32 [batch + 1], q and out [total, Hq, D])."""
    s = load().pkv_extend_attn(_ws(ws), int(batch), int(layer), _ptr(qo_indptr),
                               int(max_qo_len), _ptr(q), _ptr(out), float(scale),
                               int(num_splits), int(flags), _stream(stream))
    return _check("pkv_extend_attn", s) if check else s


def pkv_extend_append(ws, batch, layer, qo_indptr, max_qo_len, k_new, v_new, stream=None,
                      check=True):
    s = load().pkv_extend_append(_ws(ws), int(batch), int(layer), _ptr(qo_indptr),
                                 int(max_qo_len), _ptr(k_new), _ptr(v_new), _stream(stream))
    return _check("pkv_extend_append", s) if check else s


def pkv_merge_lse(n_rows, head_dim, o_a, lse_a, o_b, lse_b, out, lse_out=None, flags=0,
                  stream=None, check=True):
    """Log-sum-exp merge of two results over disjoint keys of the same rows."""
    s = load().pkv_merge_lse(int(n_rows), int(head_dim), _ptr(o_a), _ptr(lse_a), _ptr(o_b),
                             _ptr(lse_b), _ptr(out), _ptr(lse_out), int(flags), _stream(stream))
    return _check("pkv_merge_lse", s) if check else s


def pkv_is_steady_increment(prev_ids, prev_lens, ids, lens) -> bool:
    """Host arrays (sequences of ints); see include/pkv.h."""
    if prev_ids is None or prev_lens is None:
        return False
    n_prev, n = len(prev_ids), len(ids)
    A64 = ctypes.c_int64 * max(1, n_prev)
    A32 = ctypes.c_int32 * max(1, n_prev)
    B64 = ctypes.c_int64 * max(1, n)
    B32 = ctypes.c_int32 * max(1, n)
    r = load().pkv_is_steady_increment(A64(*prev_ids), A32(*prev_lens), n_prev, B64(*ids),
                                       B32(*lens), n)
    return bool(r)
