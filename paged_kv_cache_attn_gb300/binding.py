"""Thin ctypes binding of ``libpagedkv.so`` (the C ABI in ``include/pagedkv.h``).

Argument marshalling only: every function here has the name of the C entry
point it calls, turns torch tensors / numpy arrays into pointers and raises
:class:`KVError` on a non-zero status.  No step of the decode path runs in
Python.  The library must have been built (``__graft_entry__.build()`` or
``python -m paged_kv_cache_attn_gb300.build``); importing this module without
it raises ImportError -- there is no fallback.
"""

from __future__ import annotations

import ctypes as C
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libpagedkv.so")

KV_OK = 0
KV_ERR_OOM = 1
KV_ERR_INVALID_ARG = 2
KV_ERR_NOT_FOUND = 3
KV_ERR_CUDA = 4
KV_ERR_DEVICE = 5
KV_ERR_TIMEOUT = 6
KV_ERR_INTERNAL = 7
KV_STOP_FREE_BLOCKS = 0
KV_STOP_EVICTED_LEAVES = 1
KV_PLAN_NO_TENSOR_CORES = 1
KV_PLAN_IGNORE_GROUPS = 2
KV_PLAN_KV_E4M3 = 4
KV_PLAN_NARROW_TILES = 8
KV_DTYPE_BF16 = 0
KV_DTYPE_E4M3 = 1

_NAMES = {0: "OK", 1: "OOM", 2: "INVALID_ARG", 3: "NOT_FOUND", 4: "CUDA",
          5: "DEVICE", 6: "TIMEOUT", 7: "INTERNAL"}


class KVError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{_NAMES.get(code, code)}: {msg}")
        self.code = code


class kv_pool_desc(C.Structure):
    _fields_ = [("num_blocks", C.c_int64), ("block_size", C.c_int32),
                ("num_layers", C.c_int32), ("num_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("k_pool", C.c_void_p),
                ("v_pool", C.c_void_p),
                ("initial_free_order", C.POINTER(C.c_int32)),
                ("kv_dtype", C.c_int32), ("kv_scales", C.c_void_p)]


class kv_branch_info_t(C.Structure):
    _fields_ = [("live", C.c_int32), ("parent", C.c_int32),
                ("depth", C.c_int32), ("seq_len", C.c_int32),
                ("n_blocks", C.c_int32), ("n_children", C.c_int32)]


class kv_decode_plan_info(C.Structure):
    _fields_ = [("plan_ints", C.c_int64), ("workspace_bytes", C.c_int64),
                ("partial_rows", C.c_int64), ("n_row_items", C.c_int32),
                ("n_tile_items", C.c_int32), ("n_merge_rows", C.c_int32),
                ("chunk_blocks", C.c_int32), ("n_tile_wide_items", C.c_int32),
                ("flags", C.c_int32), ("n_row_warp_items", C.c_int32),
                ("reserved", C.c_int32)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class kv_radix_node_t(C.Structure):
    _fields_ = [("live", C.c_int32), ("parent", C.c_int32),
                ("n_blocks", C.c_int32), ("lock_ref", C.c_int32),
                ("n_children", C.c_int32), ("reserved", C.c_int32),
                ("last_access", C.c_int64)]


_i32p = C.POINTER(C.c_int32)
_i64p = C.POINTER(C.c_int64)
_f64p = C.POINTER(C.c_double)
_vp = C.c_void_p

# name -> (restype, argtypes)
_SIGS = {
    "kv_pool_create": (C.c_int32, [C.POINTER(kv_pool_desc), C.POINTER(_vp)]),
    "kv_pool_destroy": (C.c_int32, [_vp]),
    "kv_branch_create": (C.c_int32, [_vp, _i32p]),
    "kv_append": (C.c_int32, [_vp, C.c_int32, C.c_int32, _vp, _vp, _vp]),
    "kv_fork_branch": (C.c_int32, [_vp, C.c_int32, _i32p, _vp]),
    "kv_fork_branches": (C.c_int32, [_vp, C.c_int32, C.c_int32, _i32p, _vp]),
    "kv_append_batch": (C.c_int32, [_vp, C.c_int32, _i32p, _i32p, _vp, _vp,
                                    _vp]),
    "kv_reserve": (C.c_int32, [_vp, C.c_int32, _i32p, _i32p]),
    "kv_free": (C.c_int32, [_vp, C.c_int32]),
    "kv_free_subtree": (C.c_int32, [_vp, C.c_int32, _i32p, _i32p]),
    "kv_evict_order": (C.c_int32, [_vp, C.c_int32, _i32p, _f64p, _i32p]),
    "kv_evict": (C.c_int32, [_vp, C.c_int32, _i32p, _f64p, C.c_int32,
                             C.c_int64, _i32p, _i32p]),
    "kv_branch_info": (C.c_int32, [_vp, C.c_int32,
                                   C.POINTER(kv_branch_info_t)]),
    "kv_get_block_table": (C.c_int32, [_vp, C.c_int32, _i32p, C.c_int32,
                                       _i32p, _i32p]),
    "kv_get_refcounts": (C.c_int32, [_vp, _i32p]),
    "kv_get_free_stack": (C.c_int32, [_vp, _i32p, C.c_int64, _i64p]),
    "kv_num_branches": (C.c_int32, [_vp, _i32p]),
    "kv_bytes_per_token": (C.c_int64, [C.c_int32] * 4),
    "kv_batch_max_blocks": (C.c_int32, [_vp, C.c_int32, _i32p, _i32p]),
    "kv_build_batch": (C.c_int32, [_vp, C.c_int32, _i32p, C.c_int32, _i32p,
                                   _i32p, C.c_int32, _i32p, _i32p]),
    "paged_decode_plan": (C.c_int32, [C.c_int32] * 6 +
                          [_i32p, _i32p, C.c_int32, C.c_int32, C.c_int32,
                           _i32p, C.c_int64,
                           C.POINTER(kv_decode_plan_info)]),
    "paged_decode_attn_workspace_size": (
        C.c_int32, [C.POINTER(kv_decode_plan_info), C.POINTER(C.c_size_t)]),
    "paged_decode_attn": (C.c_int32, [_vp, _vp, _vp, C.c_int64, _vp, _vp, _vp,
                                      C.c_int32, C.c_int32, C.c_int32,
                                      C.c_int32, C.c_int32, C.c_int32,
                                      C.c_int32, C.c_float, _vp, _vp,
                                      C.POINTER(kv_decode_plan_info), _vp,
                                      C.c_size_t, _vp]),
    "paged_decode_append_attn": (C.c_int32, [_vp, _vp, _vp, _vp, _vp,
                                             C.c_int64, _vp, _vp, _vp,
                                             C.c_int32, C.c_int32, C.c_int32,
                                             C.c_int32, C.c_int32, C.c_int32,
                                             C.c_int32, C.c_float, _vp, _vp,
                                             C.POINTER(kv_decode_plan_info),
                                             _vp, C.c_size_t, _vp]),
    "paged_decode_attn_noalloc": (C.c_int32, [_vp, _vp, _vp, C.c_int64, _vp,
                                              _vp, _vp, C.c_int32, C.c_int32,
                                              C.c_int32, C.c_int32, C.c_int32,
                                              C.c_int32, C.c_int32, C.c_float,
                                              _vp, _vp,
                                              C.POINTER(kv_decode_plan_info),
                                              _vp]),
    "kv_check_noalloc_status": (C.c_int32, [_vp, C.POINTER(C.c_int32),
                                            C.POINTER(C.c_int32)]),
    "paged_decode_attn_e4m3": (C.c_int32, [_vp, _vp, _vp, _vp, C.c_int64, _vp,
                                           _vp, _vp, C.c_int32, C.c_int32,
                                           C.c_int32, C.c_int32, C.c_int32,
                                           C.c_int32, C.c_int32, C.c_float,
                                           _vp, _vp,
                                           C.POINTER(kv_decode_plan_info),
                                           _vp, C.c_size_t, _vp]),
    "paged_decode_append_attn_e4m3": (C.c_int32, [_vp, _vp, _vp, _vp, _vp, _vp,
                                                  C.c_int64, _vp, _vp, _vp,
                                                  C.c_int32, C.c_int32,
                                                  C.c_int32, C.c_int32,
                                                  C.c_int32, C.c_int32,
                                                  C.c_int32, C.c_float, _vp,
                                                  _vp,
                                                  C.POINTER(kv_decode_plan_info),
                                                  _vp, C.c_size_t, _vp]),
    "kv_check_device_status": (C.c_int32, [_vp, _vp, _i32p, _i32p]),
    "kv_selftest_timeout": (C.c_int32, [_vp, C.c_int64, _vp]),
    "kv_offload_attach": (C.c_int32, [_vp, _vp, _vp, _vp, C.c_int64]),
    "kv_spill": (C.c_int32, [_vp, C.c_int32, _i32p, _vp, _i32p]),
    "kv_restore": (C.c_int32, [_vp, C.c_int32, _i32p, _vp, _i32p]),
    "kv_get_host_free": (C.c_int32, [_vp, _i32p, C.c_int64, _i64p]),
    "kv_radix_create": (C.c_int32, [_vp, C.POINTER(_vp)]),
    "kv_radix_destroy": (C.c_int32, [_vp]),
    "kv_radix_match": (C.c_int32, [_vp, C.c_int32, _i32p, _i32p, _i32p]),
    "kv_radix_insert": (C.c_int32, [_vp, C.c_int32, C.c_int32, _i32p, _i32p]),
    "kv_radix_fork": (C.c_int32, [_vp, C.c_int32, _i32p]),
    "kv_radix_lock": (C.c_int32, [_vp, C.c_int32]),
    "kv_radix_unlock": (C.c_int32, [_vp, C.c_int32]),
    "kv_radix_evict": (C.c_int32, [_vp, C.c_int64, _i32p, _i32p]),
    "kv_radix_node_info": (C.c_int32, [_vp, C.c_int32,
                                       C.POINTER(kv_radix_node_t)]),
    "kv_radix_node_blocks": (C.c_int32, [_vp, C.c_int32, _i32p, C.c_int32,
                                         _i32p]),
    "kv_radix_num_nodes": (C.c_int32, [_vp, _i32p]),
    "kv_set_launch_events": (C.c_int32, [C.POINTER(_vp), C.c_int32]),
    "kv_last_error": (C.c_char_p, []),
}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run "
                          "`python -m paged_kv_cache_attn_gb300.build` or "
                          "__graft_entry__.build() first")
    lib = C.CDLL(LIB_PATH)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()
EXPORTED = tuple(_SIGS)


def lib():
    return _lib


def _check(status: int) -> None:
    if status != KV_OK:
        raise KVError(status, _lib.kv_last_error().decode())


def _ptr(x):
    """Device/host pointer of a torch tensor, numpy array, int or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream if \
            torch.cuda.is_available() else None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _as_i32p(a: np.ndarray):
    return a.ctypes.data_as(_i32p)


# ---- pool lifetime -------------------------------------------------------------

def kv_pool_create(num_blocks, num_layers, num_kv_heads, head_dim,
                   k_pool=None, v_pool=None, initial_free_order=None,
                   block_size=16, kv_dtype=KV_DTYPE_BF16, kv_scales=None):
    order = None if initial_free_order is None else _i32(initial_free_order)
    d = kv_pool_desc(num_blocks, block_size, num_layers, num_kv_heads,
                     head_dim, _ptr(k_pool), _ptr(v_pool),
                     None if order is None else _as_i32p(order), kv_dtype,
                     _ptr(kv_scales))
    h = _vp()
    _check(_lib.kv_pool_create(C.byref(d), C.byref(h)))
    return h


def kv_pool_destroy(h):
    _check(_lib.kv_pool_destroy(h))


def kv_branch_create(h) -> int:
    out = C.c_int32()
    _check(_lib.kv_branch_create(h, C.byref(out)))
    return out.value


def kv_append(h, bid, n_tokens, k_new=None, v_new=None, stream=None):
    s = _stream(stream) if k_new is not None else None
    _check(_lib.kv_append(h, bid, n_tokens, _ptr(k_new), _ptr(v_new), s))


def kv_append_batch(h, ids, n_tokens, k_new=None, v_new=None, stream=None):
    ids = _i32(ids)
    n = _i32(n_tokens)
    s = _stream(stream) if k_new is not None else None
    _check(_lib.kv_append_batch(h, len(ids), _as_i32p(ids), _as_i32p(n),
                                _ptr(k_new), _ptr(v_new), s))


def kv_reserve(h, ids, n_tokens):
    ids = _i32(ids)
    n = _i32(n_tokens)
    _check(_lib.kv_reserve(h, len(ids), _as_i32p(ids), _as_i32p(n)))


def kv_fork_branch(h, parent, stream=None) -> int:
    out = C.c_int32()
    _check(_lib.kv_fork_branch(h, parent, C.byref(out), _stream(stream)))
    return out.value


def kv_fork_branches(h, parent, n, stream=None) -> list:
    out = np.zeros(n, dtype=np.int32)
    _check(_lib.kv_fork_branches(h, parent, n, _as_i32p(out), _stream(stream)))
    return out.tolist()


def kv_free(h, bid):
    _check(_lib.kv_free(h, bid))


def kv_free_subtree(h, bid) -> list:
    total = kv_num_branches(h)
    out = np.zeros(max(total, 1), dtype=np.int32)
    n = C.c_int32()
    _check(_lib.kv_free_subtree(h, bid, C.byref(n), _as_i32p(out)))
    return out[:n.value].tolist()


def kv_evict_order(h, ids, scores) -> list:
    ids = _i32(ids)
    sc = np.ascontiguousarray(scores, dtype=np.float64)
    out = np.zeros(len(ids), dtype=np.int32)
    _check(_lib.kv_evict_order(h, len(ids), _as_i32p(ids),
                               sc.ctypes.data_as(_f64p), _as_i32p(out)))
    return out.tolist()


def kv_evict(h, ids, scores, stop_kind, target) -> list:
    ids = _i32(ids)
    sc = np.ascontiguousarray(scores, dtype=np.float64)
    out = np.zeros(max(len(ids), 1), dtype=np.int32)
    n = C.c_int32()
    _check(_lib.kv_evict(h, len(ids), _as_i32p(ids), sc.ctypes.data_as(_f64p),
                         stop_kind, target, C.byref(n), _as_i32p(out)))
    return out[:n.value].tolist()


# ---- introspection ---------------------------------------------------------------

def kv_branch_info(h, bid) -> dict:
    out = kv_branch_info_t()
    _check(_lib.kv_branch_info(h, bid, C.byref(out)))
    return {f: getattr(out, f) for f, _ in out._fields_}


def kv_get_block_table(h, bid):
    n = C.c_int32()
    L = C.c_int32()
    _check(_lib.kv_get_block_table(h, bid, None, 0, C.byref(n), C.byref(L)))
    out = np.zeros(max(n.value, 1), dtype=np.int32)
    _check(_lib.kv_get_block_table(h, bid, _as_i32p(out), n.value, C.byref(n),
                                   C.byref(L)))
    return out[:n.value], L.value


def kv_get_refcounts(h, num_blocks) -> np.ndarray:
    out = np.zeros(num_blocks, dtype=np.int32)
    _check(_lib.kv_get_refcounts(h, _as_i32p(out)))
    return out


def kv_get_free_stack(h) -> np.ndarray:
    n = C.c_int64()
    _check(_lib.kv_get_free_stack(h, None, 0, C.byref(n)))
    out = np.zeros(max(n.value, 1), dtype=np.int32)
    _check(_lib.kv_get_free_stack(h, _as_i32p(out), n.value, C.byref(n)))
    return out[:n.value]


def kv_num_branches(h) -> int:
    out = C.c_int32()
    _check(_lib.kv_num_branches(h, C.byref(out)))
    return out.value


def kv_bytes_per_token(num_layers, num_heads, head_dim, elem_bytes) -> int:
    return _lib.kv_bytes_per_token(num_layers, num_heads, head_dim, elem_bytes)


# ---- decode batch and attention ------------------------------------------------

def kv_batch_max_blocks(h, ids) -> int:
    ids = _i32(ids)
    out = C.c_int32()
    _check(_lib.kv_batch_max_blocks(h, len(ids), _as_i32p(ids), C.byref(out)))
    return out.value


def kv_build_batch(h, ids, max_blocks=None, tables=None, seq_lens=None,
                   groups=None):
    """Host (tables [nb][max_blocks], seq_lens [nb], groups [ng][4]).

    Optional output arrays (int32, C-contiguous; groups with >= nb rows of 4)
    are filled in place -- e.g. numpy views of pinned staging buffers; the
    returned groups is then a view of the filled rows."""
    ids = _i32(ids)
    nb = len(ids)
    if max_blocks is None:
        max_blocks = max(kv_batch_max_blocks(h, ids), 1)
    if tables is None:
        tables = np.zeros((nb, max_blocks), dtype=np.int32)
    if seq_lens is None:
        seq_lens = np.zeros(nb, dtype=np.int32)
    fresh = groups is None
    if fresh:
        groups = np.zeros((nb + 1, 4), dtype=np.int32)
    for a in (tables, seq_lens, groups):
        assert a.dtype == np.int32 and a.flags.c_contiguous
    assert tables.size >= nb * max_blocks and seq_lens.size >= nb
    ng = C.c_int32()
    _check(_lib.kv_build_batch(h, nb, _as_i32p(ids), max_blocks,
                               _as_i32p(tables), _as_i32p(seq_lens),
                               groups.size // 4, C.byref(ng),
                               _as_i32p(groups)))
    g = groups.reshape(-1, 4)[:ng.value]
    return tables, seq_lens, (g.copy() if fresh else g)


def paged_decode_plan(nb, Hq, Hkv, head_dim, max_blocks, seq_lens, groups,
                      num_sms=0, flags=0, block_size=16, plan_out=None):
    """Host plan (int32 array) and its kv_decode_plan_info.  With plan_out
    (int32, large enough) the plan is written there and a view returned."""
    lens = _i32(seq_lens)
    g = _i32(groups).reshape(-1, 4)
    info = kv_decode_plan_info()
    gp = _as_i32p(g) if len(g) else None
    if plan_out is not None:
        assert plan_out.dtype == np.int32 and plan_out.flags.c_contiguous
        _check(_lib.paged_decode_plan(nb, Hq, Hkv, head_dim, block_size,
                                      max_blocks, _as_i32p(lens), gp, len(g),
                                      num_sms, flags, _as_i32p(plan_out),
                                      plan_out.size, C.byref(info)))
        return plan_out[:info.plan_ints], info
    _check(_lib.paged_decode_plan(nb, Hq, Hkv, head_dim, block_size,
                                  max_blocks, _as_i32p(lens), gp, len(g),
                                  num_sms, flags, None, 0, C.byref(info)))
    plan = np.zeros(info.plan_ints, dtype=np.int32)
    _check(_lib.paged_decode_plan(nb, Hq, Hkv, head_dim, block_size,
                                  max_blocks, _as_i32p(lens), gp, len(g),
                                  num_sms, flags, _as_i32p(plan), len(plan),
                                  C.byref(info)))
    return plan, info


def paged_decode_attn_workspace_size(info) -> int:
    out = C.c_size_t()
    _check(_lib.paged_decode_attn_workspace_size(C.byref(info), C.byref(out)))
    return out.value


def paged_decode_attn(q, k_pool, v_pool, num_blocks, block_tables, seq_lens,
                      prefix_groups, n_groups, nb, max_blocks, Hq, Hkv,
                      head_dim, scale, out, plan, info, workspace, ws_bytes,
                      stream=None, block_size=16):
    _check(_lib.paged_decode_attn(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), num_blocks, _ptr(block_tables),
        _ptr(seq_lens), _ptr(prefix_groups), n_groups, nb, max_blocks, Hq, Hkv,
        head_dim, block_size, scale, _ptr(out), _ptr(plan), C.byref(info),
        _ptr(workspace), ws_bytes, _stream(stream)))


def paged_decode_append_attn(q, k_step, v_step, k_pool, v_pool, num_blocks,
                             block_tables, seq_lens, prefix_groups, n_groups,
                             nb, max_blocks, Hq, Hkv, head_dim, scale, out,
                             plan, info, workspace, ws_bytes, stream=None,
                             block_size=16):
    _check(_lib.paged_decode_append_attn(
        _ptr(q), _ptr(k_step), _ptr(v_step), _ptr(k_pool), _ptr(v_pool),
        num_blocks, _ptr(block_tables), _ptr(seq_lens), _ptr(prefix_groups),
        n_groups, nb, max_blocks, Hq, Hkv, head_dim, block_size, scale,
        _ptr(out), _ptr(plan), C.byref(info), _ptr(workspace), ws_bytes,
        _stream(stream)))


def paged_decode_attn_e4m3(q, k_pool, v_pool, kv_scales, num_blocks,
                           block_tables, seq_lens, prefix_groups, n_groups, nb,
                           max_blocks, Hq, Hkv, head_dim, scale, out, plan,
                           info, workspace, ws_bytes, stream=None,
                           block_size=16):
    _check(_lib.paged_decode_attn_e4m3(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(kv_scales), num_blocks,
        _ptr(block_tables), _ptr(seq_lens), _ptr(prefix_groups), n_groups, nb,
        max_blocks, Hq, Hkv, head_dim, block_size, scale, _ptr(out),
        _ptr(plan), C.byref(info), _ptr(workspace), ws_bytes, _stream(stream)))


def paged_decode_append_attn_e4m3(q, k_step, v_step, k_pool, v_pool,
                                  kv_scales, num_blocks, block_tables,
                                  seq_lens, prefix_groups, n_groups, nb,
                                  max_blocks, Hq, Hkv, head_dim, scale, out,
                                  plan, info, workspace, ws_bytes,
                                  stream=None, block_size=16):
    _check(_lib.paged_decode_append_attn_e4m3(
        _ptr(q), _ptr(k_step), _ptr(v_step), _ptr(k_pool), _ptr(v_pool),
        _ptr(kv_scales), num_blocks, _ptr(block_tables), _ptr(seq_lens),
        _ptr(prefix_groups), n_groups, nb, max_blocks, Hq, Hkv, head_dim,
        block_size, scale, _ptr(out), _ptr(plan), C.byref(info),
        _ptr(workspace), ws_bytes, _stream(stream)))


def paged_decode_attn_noalloc(q, k_pool, v_pool, num_blocks, block_tables,
                              seq_lens, prefix_groups, n_groups, nb,
                              max_blocks, Hq, Hkv, head_dim, scale, out, plan,
                              info, stream=None, block_size=16):
    """paged_decode_attn with the library's built-in scratch (no workspace)."""
    _check(_lib.paged_decode_attn_noalloc(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), num_blocks, _ptr(block_tables),
        _ptr(seq_lens), _ptr(prefix_groups), n_groups, nb, max_blocks, Hq, Hkv,
        head_dim, block_size, scale, _ptr(out), _ptr(plan), C.byref(info),
        _stream(stream)))


def kv_check_noalloc_status(stream=None):
    """(code, detail) of the built-in scratch's status word on the current
    device, read and cleared."""
    code = C.c_int32()
    detail = C.c_int32()
    _check(_lib.kv_check_noalloc_status(_stream(stream), C.byref(code),
                                        C.byref(detail)))
    return code.value, detail.value


def kv_selftest_timeout(workspace, wait_cycles, stream=None):
    _check(_lib.kv_selftest_timeout(_ptr(workspace), wait_cycles,
                                    _stream(stream)))


def kv_check_device_status(workspace, stream=None):
    code = C.c_int32()
    detail = C.c_int32()
    _check(_lib.kv_check_device_status(_ptr(workspace), _stream(stream),
                                       C.byref(code), C.byref(detail)))
    return code.value, detail.value


_events_keepalive = None


def kv_set_launch_events(events):
    """events: list of 6 torch.cuda.Event (created with enable_timing) or
    None to clear."""
    global _events_keepalive
    if not events:
        _events_keepalive = None
        _check(_lib.kv_set_launch_events(None, 0))
        return
    handles = [e.cuda_event if e is not None else None for e in events]
    if any(e is not None and not h for e, h in zip(events, handles)):
        raise ValueError("record each torch.cuda.Event once before passing it "
                         "(torch creates the CUDA event on first record)")
    arr = (_vp * len(events))(*handles)
    _events_keepalive = arr
    _check(_lib.kv_set_launch_events(arr, len(events)))


# ---- radix prefix index ------------------------------------------------------

def kv_radix_create(pool):
    h = _vp()
    _check(_lib.kv_radix_create(pool, C.byref(h)))
    return h


def kv_radix_destroy(r):
    _check(_lib.kv_radix_destroy(r))


def kv_radix_match(r, tokens):
    t = _i32(tokens)
    node, n = C.c_int32(), C.c_int32()
    _check(_lib.kv_radix_match(r, len(t), _as_i32p(t) if len(t) else None,
                               C.byref(node), C.byref(n)))
    return node.value, n.value


def kv_radix_insert(r, branch, tokens):
    t = _i32(tokens)
    node = C.c_int32()
    _check(_lib.kv_radix_insert(r, branch, len(t),
                                _as_i32p(t) if len(t) else None,
                                C.byref(node)))
    return node.value


def kv_radix_fork(r, node):
    out = C.c_int32()
    _check(_lib.kv_radix_fork(r, node, C.byref(out)))
    return out.value


def kv_radix_lock(r, node):
    _check(_lib.kv_radix_lock(r, node))


def kv_radix_unlock(r, node):
    _check(_lib.kv_radix_unlock(r, node))


def kv_radix_num_nodes(r):
    out = C.c_int32()
    _check(_lib.kv_radix_num_nodes(r, C.byref(out)))
    return out.value


def kv_radix_evict(r, target_free_blocks):
    cap = max(kv_radix_num_nodes(r), 1)
    out = np.zeros(cap, dtype=np.int32)
    n = C.c_int32()
    _check(_lib.kv_radix_evict(r, target_free_blocks, C.byref(n),
                               _as_i32p(out)))
    return out[:n.value].tolist()


def kv_radix_node_info(r, node):
    out = kv_radix_node_t()
    _check(_lib.kv_radix_node_info(r, node, C.byref(out)))
    return {f: getattr(out, f) for f, _ in out._fields_ if f != "reserved"}


def kv_radix_node_blocks(r, node):
    n = C.c_int32()
    _check(_lib.kv_radix_node_blocks(r, node, None, 0, C.byref(n)))
    out = np.zeros(max(n.value, 1), dtype=np.int32)
    _check(_lib.kv_radix_node_blocks(r, node, _as_i32p(out), n.value,
                                     C.byref(n)))
    return out[:n.value].tolist()


# ---- host tier ----------------------------------------------------------------

def kv_offload_attach(h, host_k, host_v, host_slots, host_scales=None):
    _check(_lib.kv_offload_attach(h, _ptr(host_k), _ptr(host_v),
                                  _ptr(host_scales), host_slots))


def kv_spill(h, ids, stream=None) -> int:
    ids = _i32(ids)
    n = C.c_int32()
    _check(_lib.kv_spill(h, len(ids), _as_i32p(ids), _stream(stream),
                         C.byref(n)))
    return n.value


def kv_restore(h, ids, stream=None) -> int:
    ids = _i32(ids)
    n = C.c_int32()
    _check(_lib.kv_restore(h, len(ids), _as_i32p(ids), _stream(stream),
                           C.byref(n)))
    return n.value


def kv_get_host_free(h) -> np.ndarray:
    n = C.c_int64()
    _check(_lib.kv_get_host_free(h, None, 0, C.byref(n)))
    out = np.zeros(max(n.value, 1), dtype=np.int32)
    _check(_lib.kv_get_host_free(h, _as_i32p(out), n.value, C.byref(n)))
    return out[:n.value]
