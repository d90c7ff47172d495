"""CPU oracle for the HiSparse KV-row swap-in and the indexed KV-row movers.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package.  The product
path (``sparse_attention_kv_row_gb300``) never imports it and shares no code
with it.

The arithmetic lives in ``hs_oracle.cpp`` (plain single-threaded C++17).  This
module only marshals numpy arrays (all host memory) into that library.

Parity status: every function here is pinned by the ``-m "not gpu"`` tests
(brute force on tiny inputs, a hand-worked example, closed forms, a textbook
LRU cache at top_k = 1, invariants, numpy index assignment for the movers, and
planted-mistake checks).  Nothing is left unpinned.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

ST_DUP_ID = 1
ST_BAD_POOL_ROW = 2
ST_BAD_LRU_SLOT = 4
ST_BAD_HOT_ROW = 8
ST_TIMEOUT = 16
ST_BAD_STATE = 32
ST_BAD_INDEX = 64


class _SwapInArgs(C.Structure):
    _fields_ = [
        ("batch", C.c_int32), ("top_k", C.c_int32), ("hot_size", C.c_int32),
        ("num_real", C.c_int32),
        ("topk_ids", C.c_void_p), ("topk_stride", C.c_int64),
        ("seq_lens", C.c_void_p), ("req_state", C.c_void_p), ("num_states", C.c_int64),
        ("slot_tokens", C.c_void_p), ("slot_tokens_stride", C.c_int64),
        ("slot_rows", C.c_void_p), ("slot_rows_stride", C.c_int64),
        ("lru", C.c_void_p), ("lru_stride", C.c_int64),
        ("pool_rows", C.c_void_p), ("pool_rows_stride", C.c_int64),
        ("pool_rows_cols", C.c_int64),
        ("pool_k", C.c_void_p), ("pool_v", C.c_void_p), ("pool_num_rows", C.c_int64),
        ("hot_k", C.c_void_p), ("hot_v", C.c_void_p), ("hot_num_rows", C.c_int64),
        ("row_bytes", C.c_int64),
        ("out_rows", C.c_void_p), ("out_stride", C.c_int64),
        ("miss_count", C.c_void_p), ("stats", C.c_void_p), ("status", C.c_void_p),
        ("miss_src", C.c_void_p), ("miss_dst", C.c_void_p), ("plan_stride", C.c_int64),
        ("miss_mask", C.c_void_p), ("mask_stride", C.c_int64),
        ("src_bt", C.c_void_p), ("src_bt_stride", C.c_int64), ("src_bt_blocks", C.c_int32),
        ("src_block_size", C.c_int32),
        ("res_bt", C.c_void_p), ("res_bt_stride", C.c_int64), ("res_bt_blocks", C.c_int32),
        ("res_block_size", C.c_int32), ("res_null_block", C.c_int32),
        ("max_seq_len", C.c_int64),
    ]


_LIBS: dict[int, C.CDLL] = {}


def load(mutant: int = 0) -> C.CDLL:
    """Build (if needed) and load the oracle library; ``mutant`` selects a
    planted-mistake build used only by the pin tests."""
    if mutant not in _LIBS:
        lib = C.CDLL(_build.build(mutant))
        lib.hso_swap_in.argtypes = [C.POINTER(_SwapInArgs)]
        lib.hso_swap_in.restype = C.c_int
        lib.hso_store_kv.argtypes = [C.c_void_p, C.c_void_p, C.c_int64, C.c_int64,
                                     C.c_void_p, C.c_void_p, C.c_int64, C.c_int64,
                                     C.c_void_p, C.c_int64, C.c_int64, C.c_void_p]
        lib.hso_store_kv.restype = C.c_int
        lib.hso_transfer_kv.argtypes = [C.c_void_p, C.c_void_p, C.c_int32, C.c_int32,
                                        C.c_void_p, C.c_void_p, C.c_int64, C.c_int64,
                                        C.c_int64, C.c_int64, C.c_int64, C.c_int64,
                                        C.c_void_p]
        lib.hso_transfer_kv.restype = C.c_int
        lib.hso_gather_misses.argtypes = [C.c_void_p, C.c_void_p, C.c_int64, C.c_void_p,
                                          C.c_void_p, C.c_int64, C.c_int64, C.c_void_p,
                                          C.c_void_p, C.c_int64, C.c_void_p, C.c_int32,
                                          C.c_int32, C.c_void_p]
        lib.hso_gather_misses.restype = C.c_int
        lib.hso_invalidate_tokens.argtypes = [C.c_void_p, C.c_int64, C.c_int32, C.c_int64,
                                              C.c_void_p, C.c_void_p, C.c_int64, C.c_void_p]
        lib.hso_invalidate_tokens.restype = C.c_int
        lib.hso_e4m3_encode_array.argtypes = [C.c_void_p, C.c_void_p, C.c_int64]
        lib.hso_e4m3_encode_array.restype = None
        lib.hso_fp8_store_kv.argtypes = [C.c_void_p, C.c_void_p, C.c_int32, C.c_int64,
                                         C.c_int64, C.c_int64, C.c_int64, C.c_void_p,
                                         C.c_void_p, C.c_int64, C.c_int64, C.c_int64,
                                         C.c_int32, C.c_int64, C.c_void_p, C.c_int64,
                                         C.c_int32, C.c_int32, C.c_void_p, C.c_void_p,
                                         C.c_void_p]
        lib.hso_fp8_store_kv.restype = C.c_int
        _LIBS[mutant] = lib
    return _LIBS[mutant]


def _ptr(a):
    return None if a is None else a.ctypes.data


def _row_stride(a: np.ndarray) -> int:
    assert a.ndim == 2 and a.strides[1] == a.itemsize, "rows must be contiguous"
    return a.strides[0] // a.itemsize


def _check(a, dtype, name, ndim=None):
    if a is None:
        return
    if a.dtype != dtype:
        raise TypeError(f"{name} must be {np.dtype(dtype).name}, got {a.dtype}")
    if ndim is not None and a.ndim != ndim:
        raise ValueError(f"{name} must be {ndim}-D")


def swap_in(*, topk_ids, seq_lens, req_state, slot_tokens, slot_rows, lru, pool_rows,
            pool_k, hot_k, out_rows, hot_size, pool_v=None, hot_v=None, num_real=-1,
            miss_count=None, stats=None, status=None, miss_src=None, miss_dst=None,
            miss_mask=None, src_block_table=None, src_block_size=1, res_block_table=None,
            res_block_size=1, res_null_block=-1, max_seq_len=0, mutant: int = 0) -> None:
    """One swap-in call over B batch rows; mutates slot_tokens, lru, hot_k/hot_v,
    out_rows and the optional outputs in place (all numpy, host memory).

    Layouts: topk_ids int32 [B,K]; seq_lens, req_state int64 [B];
    slot_tokens / slot_rows int32 [R, >=H+1]; lru int16 [R, >=H];
    pool_rows int64 [R, cols]; pool_k/pool_v uint8 [P, S];
    hot_k/hot_v uint8 [rows, S]; out_rows int32 [B, K].
    Optional plan outputs: miss_src int64 [B, >=K] and miss_dst int32 [B, >=K]
    (the row's misses in order; entries past the miss count untouched),
    miss_mask int32 [B, >=K].
    Optional block tables int32 [R, blocks]: ``src_block_table`` maps token t to
    pool row bt[r][t // bs] * bs + t % bs (entries <= 0 unmapped) in place of
    pool_rows; ``res_block_table`` serves tokens of resident blocks directly.
    """
    _check(topk_ids, np.int32, "topk_ids", 2)
    _check(seq_lens, np.int64, "seq_lens", 1)
    _check(req_state, np.int64, "req_state", 1)
    _check(slot_tokens, np.int32, "slot_tokens", 2)
    _check(slot_rows, np.int32, "slot_rows", 2)
    _check(lru, np.int16, "lru", 2)
    if pool_rows is not None:
        _check(pool_rows, np.int64, "pool_rows", 2)
    _check(src_block_table, np.int32, "src_block_table", 2)
    _check(res_block_table, np.int32, "res_block_table", 2)
    for n, a in (("pool_k", pool_k), ("pool_v", pool_v), ("hot_k", hot_k), ("hot_v", hot_v)):
        _check(a, np.uint8, n, 2)
    _check(out_rows, np.int32, "out_rows", 2)
    _check(miss_count, np.int32, "miss_count", 1)
    _check(stats, np.uint64, "stats", 1)
    _check(status, np.int32, "status", 1)
    _check(miss_src, np.int64, "miss_src", 2)
    _check(miss_dst, np.int32, "miss_dst", 2)
    _check(miss_mask, np.int32, "miss_mask", 2)
    if (miss_src is None) != (miss_dst is None):
        raise ValueError("miss_src and miss_dst go together")
    if miss_src is not None and _row_stride(miss_src) != _row_stride(miss_dst):
        raise ValueError("miss_src and miss_dst need the same row stride")
    for a in (seq_lens, req_state, pool_k, pool_v, hot_k, hot_v, miss_count, stats, status):
        if a is not None:
            assert a.flags.c_contiguous
    B, K = topk_ids.shape
    a = _SwapInArgs(
        batch=B, top_k=K, hot_size=hot_size, num_real=num_real,
        topk_ids=_ptr(topk_ids), topk_stride=_row_stride(topk_ids),
        seq_lens=_ptr(seq_lens), req_state=_ptr(req_state), num_states=slot_tokens.shape[0],
        slot_tokens=_ptr(slot_tokens), slot_tokens_stride=_row_stride(slot_tokens),
        slot_rows=_ptr(slot_rows), slot_rows_stride=_row_stride(slot_rows),
        lru=_ptr(lru), lru_stride=_row_stride(lru),
        pool_rows=_ptr(pool_rows),
        pool_rows_stride=_row_stride(pool_rows) if pool_rows is not None else 0,
        pool_rows_cols=pool_rows.shape[1] if pool_rows is not None else 0,
        pool_k=_ptr(pool_k), pool_v=_ptr(pool_v), pool_num_rows=pool_k.shape[0],
        hot_k=_ptr(hot_k), hot_v=_ptr(hot_v), hot_num_rows=hot_k.shape[0],
        row_bytes=pool_k.shape[1],
        out_rows=_ptr(out_rows), out_stride=_row_stride(out_rows),
        miss_count=_ptr(miss_count), stats=_ptr(stats), status=_ptr(status),
        miss_src=_ptr(miss_src), miss_dst=_ptr(miss_dst),
        plan_stride=_row_stride(miss_src) if miss_src is not None else 0,
        miss_mask=_ptr(miss_mask),
        mask_stride=_row_stride(miss_mask) if miss_mask is not None else 0,
        src_bt=_ptr(src_block_table),
        src_bt_stride=_row_stride(src_block_table) if src_block_table is not None else 0,
        src_bt_blocks=src_block_table.shape[1] if src_block_table is not None else 0,
        src_block_size=src_block_size,
        res_bt=_ptr(res_block_table),
        res_bt_stride=_row_stride(res_block_table) if res_block_table is not None else 0,
        res_bt_blocks=res_block_table.shape[1] if res_block_table is not None else 0,
        res_block_size=res_block_size, res_null_block=res_null_block,
        max_seq_len=max_seq_len)
    if pool_rows is None and src_block_table is None:
        raise ValueError("need pool_rows or src_block_table")
    rc = load(mutant).hso_swap_in(C.byref(a))
    if rc != 0:
        raise ValueError("oracle swap_in rejected its arguments")


def invalidate_tokens(*, slot_tokens, hot_size, state_rows, tokens, status=None) -> None:
    """Slots [0, hot_size) of state row state_rows[n] holding token tokens[n] become -1."""
    _check(slot_tokens, np.int32, "slot_tokens", 2)
    _check(state_rows, np.int64, "state_rows", 1)
    _check(tokens, np.int32, "tokens", 1)
    rc = load().hso_invalidate_tokens(_ptr(slot_tokens), _row_stride(slot_tokens), hot_size,
                                      slot_tokens.shape[0], _ptr(state_rows), _ptr(tokens),
                                      tokens.shape[0], _ptr(status))
    if rc != 0:
        raise ValueError("oracle invalidate_tokens rejected its arguments")


def gather_misses(*, pool_k, hot_k, miss_src, miss_dst, miss_count, pool_v=None, hot_v=None,
                  status=None, mutant: int = 0) -> None:
    """Replay a swap-in's miss plan onto another layer: hot row miss_dst[b][m] =
    pool row miss_src[b][m] for m < miss_count[b] (K, and V when given)."""
    for n, a in (("pool_k", pool_k), ("pool_v", pool_v), ("hot_k", hot_k), ("hot_v", hot_v)):
        _check(a, np.uint8, n, 2)
    _check(miss_src, np.int64, "miss_src", 2)
    _check(miss_dst, np.int32, "miss_dst", 2)
    _check(miss_count, np.int32, "miss_count", 1)
    if _row_stride(miss_src) != _row_stride(miss_dst):
        raise ValueError("miss_src and miss_dst need the same row stride")
    B, K = miss_src.shape
    rc = load(mutant).hso_gather_misses(
        _ptr(pool_k), _ptr(pool_v), pool_k.shape[0], _ptr(hot_k), _ptr(hot_v), hot_k.shape[0],
        pool_k.shape[1], _ptr(miss_src), _ptr(miss_dst), _row_stride(miss_src),
        _ptr(miss_count), B, K, _ptr(status))
    if rc != 0:
        raise ValueError("oracle gather_misses rejected its arguments")


_IN_DTYPES = {np.dtype(np.float32): 0, np.dtype(np.float16): 1}
IN_BF16 = 2  # bf16 inputs are passed as uint16 arrays of their bits


def e4m3_encode(x, mutant: int = 0) -> np.ndarray:
    """FP8 E4M3 codes (uint8) of float32 values: round to nearest even,
    saturating to +-448, NaN -> 0x7F with the input's sign."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    load(mutant).hso_e4m3_encode_array(_ptr(x), _ptr(out), x.size)
    return out


def fp8_store_kv(*, k, v, k_cache, v_cache, loc, page_size, k_scale=None, v_scale=None,
                 bf16=False, status=None, mutant: int = 0) -> None:
    """Quantise k/v [T, heads, dim] to FP8 E4M3 and scatter token t to slot loc[t] of
    the paged caches (uint8 [pages, page_size, heads, dim] or [slots, heads, dim]).
    ``bf16``: k and v are uint16 arrays holding bfloat16 bits.  k_scale / v_scale
    are float32 scalars (None: no scaling); values are multiplied by fp32(1/scale)."""
    if bf16:
        _check(k, np.uint16, "k", 3)
        dt = IN_BF16
    else:
        dt = _IN_DTYPES[k.dtype]
    if v is not None and v.dtype != k.dtype:
        raise TypeError("k and v must have the same dtype")
    for n, a in (("k_cache", k_cache), ("v_cache", v_cache)):
        _check(a, np.uint8, n)
    _check(loc, np.int64, "loc", 1)
    T, Hh, D = k.shape
    for a in (k, v):
        if a is not None and (a.strides[2] != a.itemsize or a.shape != k.shape):
            raise ValueError("k/v need shape [T, heads, dim] with contiguous dims")
    cs = k_cache.strides
    if k_cache.ndim == 4:
        c_page, c_off, c_head = cs[0], cs[1], cs[2]
        num_slots = k_cache.shape[0] * k_cache.shape[1]
        if k_cache.shape[1] != page_size:
            raise ValueError("page_size mismatch")
    else:
        c_page, c_off, c_head = cs[0] * page_size, cs[0], cs[1]
        num_slots = k_cache.shape[0] // page_size * page_size
    if v_cache is not None and v_cache.strides != k_cache.strides:
        raise ValueError("k_cache and v_cache need the same layout")
    ik = np.array([k_scale], np.float32) if k_scale is not None else None
    iv = np.array([v_scale], np.float32) if v_scale is not None else None
    it = k.itemsize
    rc = load(mutant).hso_fp8_store_kv(
        _ptr(k), _ptr(v), dt, k.strides[0] // it, k.strides[1] // it,
        v.strides[0] // it if v is not None else 0, v.strides[1] // it if v is not None else 0,
        _ptr(k_cache), _ptr(v_cache), c_page, c_off, c_head, page_size, num_slots, _ptr(loc), T,
        Hh, D, _ptr(ik), _ptr(iv), _ptr(status))
    if rc != 0:
        raise ValueError("oracle fp8_store_kv rejected its arguments")


def store_kv(*, k_src, v_src, k_dst, v_dst, loc, status=None) -> None:
    """k_dst[loc[t]] = k_src[t] (and V) in token order; uint8 rows [n, S]."""
    for n, a in (("k_src", k_src), ("v_src", v_src), ("k_dst", k_dst), ("v_dst", v_dst)):
        _check(a, np.uint8, n, 2)
    _check(loc, np.int64, "loc", 1)
    S = k_src.shape[1]
    rc = load().hso_store_kv(
        _ptr(k_src), _ptr(v_src), k_src.strides[0],
        v_src.strides[0] if v_src is not None else 0,
        _ptr(k_dst), _ptr(v_dst), k_dst.strides[0], k_dst.shape[0],
        _ptr(loc), loc.shape[0], S, _ptr(status))
    if rc != 0:
        raise ValueError("oracle store_kv rejected its arguments")


def transfer_kv(*, src_layers, dst_layers, src_idx, dst_idx, status=None) -> None:
    """For every index pair n and every layer l (K layers, then V layers):
    dst_layers[l][dst_idx[n]] = src_layers[l][src_idx[n]]; uint8 rows [rows, S]."""
    assert len(src_layers) == len(dst_layers) and len(src_layers) > 0
    _check(src_idx, np.int64, "src_idx", 1)
    _check(dst_idx, np.int64, "dst_idx", 1)
    S = src_layers[0].shape[1]
    src_ptrs = np.array([x.ctypes.data for x in src_layers], dtype=np.uint64)
    dst_ptrs = np.array([x.ctypes.data for x in dst_layers], dtype=np.uint64)
    rc = load().hso_transfer_kv(
        _ptr(src_ptrs), _ptr(dst_ptrs), len(src_layers), 0, _ptr(src_idx), _ptr(dst_idx),
        src_idx.shape[0], src_layers[0].strides[0], dst_layers[0].strides[0],
        min(x.shape[0] for x in src_layers), min(x.shape[0] for x in dst_layers), S,
        _ptr(status))
    if rc != 0:
        raise ValueError("oracle transfer_kv rejected its arguments")


def library_path() -> str:
    return os.path.abspath(_build.lib_path())
