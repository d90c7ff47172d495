"""HiSparse decode-time KV-row swap-in and indexed KV-row movers for GB300.

Thin PyTorch binding over libhisparse (include/hisparse.h): it checks tensor
dtypes/shapes and passes raw pointers, strides and the current CUDA stream;
every step of the computation runs in the library's sm_103a kernels.  PyTorch
provides device/pinned memory and streams only.  There is no CPU fallback: if
the library is not built, importing the binding's entry points raises.

Entry points (same names as the C ABI):
  swap_in(...)       hs_swap_in      -- resolve top-k ids, LRU-assign misses,
                                        copy missing rows, emit hot-buffer rows
  store_kv(...)      hs_store_kv     -- k_dst[loc] = k_src, v_dst[loc] = v_src
  transfer_kv(...)   hs_transfer_kv  -- per-layer / all-layer indexed row copy
  probe_read(...)    hs_probe_read   -- streaming-read bandwidth probe
"""
from __future__ import annotations

import ctypes as C

import torch

from . import _capi
from ._capi import (HisparseError, SwapInArgs, ST_BAD_HOT_ROW, ST_BAD_INDEX,  # noqa: F401
                    ST_BAD_LRU_SLOT, ST_BAD_POOL_ROW, ST_BAD_STATE, ST_DUP_ID, ST_TIMEOUT)

__all__ = ["swap_in", "swap_in_args", "make_swap_in_args", "gather_misses", "fp8_store_kv",
           "invalidate_tokens", "wait_selftest", "swap_in_timeout_selftest",
           "swap_in_layers", "swap_in_layers_timeout_selftest", "layer_args_array",
           "store_kv", "transfer_kv",
           "transfer_kv_layers", "probe_read", "swap_in_smem_bytes", "library_path",
           "HisparseError", "SwapInArgs"]


def library_path() -> str:
    return _capi.LIB_PATH


def _lib():
    return _capi.load()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if isinstance(stream, torch.cuda.Stream) else int(stream)


def _ptr(t) -> int | None:
    return None if t is None else int(t.data_ptr())


def _need(t, dtype, name, ndim=None):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must be {ndim}-D, got shape {tuple(t.shape)}")
    if ndim == 2 and t.shape[1] > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} rows must be contiguous")
    if ndim == 1 and t.numel() > 1 and t.stride(0) != 1:
        raise ValueError(f"{name} must be contiguous")


def _byte_rows(t, name):
    """(ptr, rows, row_bytes, pitch_bytes) of a tensor whose trailing dims are
    one contiguous row."""
    if t.dim() < 1:
        raise ValueError(f"{name} must have a leading row axis")
    inner = t[0] if t.shape[0] > 0 else t.new_empty(t.shape[1:])
    if t.dim() > 1 and not inner.is_contiguous():
        raise ValueError(f"{name}: each row must be contiguous")
    row_bytes = (inner.numel() if t.dim() > 1 else 1) * t.element_size()
    pitch = (t.stride(0) if t.dim() > 1 else 1) * t.element_size()
    return int(t.data_ptr()), int(t.shape[0]), int(row_bytes), int(pitch)


def swap_in_smem_bytes(top_k: int, hot_size: int) -> int:
    return int(_lib().hs_swap_in_smem_bytes(top_k, hot_size))


def make_swap_in_args(*, topk_ids, seq_lens, req_state, slot_tokens, slot_rows, lru, pool_rows,
                      pool_k, hot_k, out_rows, hot_size=None, pool_v=None, hot_v=None,
                      num_real=None, miss_count=None, stats=None, status=None,
                      miss_src=None, miss_dst=None, miss_mask=None,
                      src_block_table=None, src_block_size=1, res_block_table=None,
                      res_block_size=1, res_null_block=-1, max_seq_len=0,
                      overlap_prev=False) -> SwapInArgs:
    """Build a reusable ``hs_swap_in_args`` for these tensors (see include/hisparse.h).

    ``overlap_prev`` sets HS_OVERLAP_PREV: the launch may start while the
    kernel before it in the stream still runs, reading only the request
    metadata and state rows (seq_lens, req_state, num_real, slot_tokens,
    slot_rows, lru) until that kernel completes.

    ``miss_src`` (int64) / ``miss_dst`` (int32) [B, >=K] receive the row's miss
    plan (pool row and hot row of each miss, in order, the first miss_count[b]
    entries) and ``miss_mask`` (int32 [B, >=K]) marks the entries that missed;
    ``gather_misses`` replays the plan onto another layer.

    ``src_block_table`` (int32 [R, blocks], pool_rows may then be None) maps token t
    to pool row bt[r][t // bs] * bs + t % bs; ``res_block_table`` serves tokens of
    resident blocks directly (see include/hisparse.h).

    ``max_seq_len`` (0 = unknown) bounds every row's sequence length; rows above it
    report HS_ST_BAD_STATE.  Giving it lets the kernel use its compact hash."""
    H = int(hot_size if hot_size is not None else lru.shape[1])
    _need(topk_ids, torch.int32, "topk_ids", 2)
    _need(out_rows, torch.int32, "out_rows", 2)
    _need(slot_tokens, torch.int32, "slot_tokens", 2)
    _need(slot_rows, torch.int32, "slot_rows", 2)
    _need(lru, torch.int16, "lru", 2)
    if pool_rows is None and src_block_table is None:
        raise ValueError("need pool_rows or src_block_table")
    if pool_rows is not None:
        _need(pool_rows, torch.int64, "pool_rows", 2)
    for t, name in ((src_block_table, "src_block_table"), (res_block_table, "res_block_table")):
        if t is not None:
            _need(t, torch.int32, name, 2)
    if seq_lens.dtype not in (torch.int32, torch.int64) or req_state.dtype not in (
            torch.int32, torch.int64):
        raise TypeError("seq_lens and req_state must be int32 or int64")
    _need(seq_lens, seq_lens.dtype, "seq_lens", 1)
    _need(req_state, req_state.dtype, "req_state", 1)
    if num_real is not None:
        _need(num_real, torch.int32, "num_real", 1)
    if miss_count is not None:
        _need(miss_count, torch.int32, "miss_count", 1)
    if status is not None:
        _need(status, torch.int32, "status", 1)
    if (miss_src is None) != (miss_dst is None):
        raise ValueError("miss_src and miss_dst go together")
    if miss_src is not None:
        _need(miss_src, torch.int64, "miss_src", 2)
        _need(miss_dst, torch.int32, "miss_dst", 2)
        if miss_src.stride(0) != miss_dst.stride(0):
            raise ValueError("miss_src and miss_dst need the same row stride")
        if miss_count is None:
            raise ValueError("the miss plan needs miss_count")
    if miss_mask is not None:
        _need(miss_mask, torch.int32, "miss_mask", 2)
    if stats is not None:
        if stats.dtype not in (torch.int64, getattr(torch, "uint64", torch.int64)) or \
                stats.numel() < 2:
            raise TypeError("stats must be a 2-element 64-bit integer tensor")
    B, K = topk_ids.shape
    if out_rows.shape[0] < B or out_rows.shape[1] < K:
        raise ValueError("out_rows must be at least [batch, top_k]")
    if seq_lens.numel() < B or req_state.numel() < B:
        raise ValueError("seq_lens and req_state need one entry per batch row")
    pk_ptr, p_rows, row_bytes, p_pitch = _byte_rows(pool_k, "pool_k")
    hk_ptr, h_rows, h_bytes, h_pitch = _byte_rows(hot_k, "hot_k")
    if h_bytes != row_bytes or p_pitch != row_bytes or h_pitch != row_bytes:
        raise ValueError("pool and hot buffers need contiguous rows of the same byte width")
    pv_ptr = hv_ptr = None
    if pool_v is not None or hot_v is not None:
        if pool_v is None or hot_v is None:
            raise ValueError("pool_v and hot_v go together")
        pv_ptr, pv_rows, pv_bytes, pv_pitch = _byte_rows(pool_v, "pool_v")
        hv_ptr, hv_rows, hv_bytes, hv_pitch = _byte_rows(hot_v, "hot_v")
        if {pv_bytes, hv_bytes, pv_pitch, hv_pitch} != {row_bytes}:
            raise ValueError("V buffers need the same row width as K")
        p_rows, h_rows = min(p_rows, pv_rows), min(h_rows, hv_rows)
    flags = (_capi.SEQ_LENS_I64 if seq_lens.dtype == torch.int64 else 0) | (
        _capi.REQ_STATE_I64 if req_state.dtype == torch.int64 else 0) | (
        _capi.OVERLAP_PREV if overlap_prev else 0)
    args = SwapInArgs(
        batch=B, top_k=K, hot_size=H, flags=flags, num_real=_ptr(num_real),
        topk_ids=_ptr(topk_ids), topk_stride=topk_ids.stride(0),
        seq_lens=_ptr(seq_lens), req_state=_ptr(req_state),
        num_states=min([slot_tokens.shape[0], slot_rows.shape[0], lru.shape[0]] +
                       [t.shape[0] for t in (pool_rows, src_block_table, res_block_table)
                        if t is not None]),
        slot_tokens=_ptr(slot_tokens), slot_tokens_stride=slot_tokens.stride(0),
        slot_rows=_ptr(slot_rows), slot_rows_stride=slot_rows.stride(0),
        lru=_ptr(lru), lru_stride=lru.stride(0),
        pool_rows=_ptr(pool_rows),
        pool_rows_stride=pool_rows.stride(0) if pool_rows is not None else 0,
        pool_rows_cols=pool_rows.shape[1] if pool_rows is not None else 0,
        pool_k=pk_ptr, pool_v=pv_ptr, pool_num_rows=p_rows,
        hot_k=hk_ptr, hot_v=hv_ptr, hot_num_rows=h_rows,
        row_bytes=row_bytes, out_rows=_ptr(out_rows), out_stride=out_rows.stride(0),
        miss_count=_ptr(miss_count), stats=_ptr(stats), status=_ptr(status),
        miss_src=_ptr(miss_src), miss_dst=_ptr(miss_dst),
        plan_stride=miss_src.stride(0) if miss_src is not None else 0,
        miss_mask=_ptr(miss_mask),
        mask_stride=miss_mask.stride(0) if miss_mask is not None else 0,
        src_bt=_ptr(src_block_table),
        src_bt_stride=src_block_table.stride(0) if src_block_table is not None else 0,
        src_bt_blocks=src_block_table.shape[1] if src_block_table is not None else 0,
        src_block_size=src_block_size,
        res_bt=_ptr(res_block_table),
        res_bt_stride=res_block_table.stride(0) if res_block_table is not None else 0,
        res_bt_blocks=res_block_table.shape[1] if res_block_table is not None else 0,
        res_block_size=res_block_size, res_null_block=res_null_block,
        max_seq_len=int(max_seq_len))
    for t, name in ((miss_src, "miss_src"), (miss_dst, "miss_dst"), (miss_mask, "miss_mask")):
        if t is not None and (t.shape[0] < B or t.shape[1] < K):
            raise ValueError(f"{name} must be at least [batch, top_k]")
    # the struct holds raw pointers: keep the tensors alive as long as it lives
    args.tensors = (topk_ids, seq_lens, req_state, slot_tokens, slot_rows, lru, pool_rows,
                    pool_k, pool_v, hot_k, hot_v, out_rows, num_real, miss_count, stats, status,
                    miss_src, miss_dst, miss_mask, src_block_table, res_block_table)
    return args


def swap_in_args(args: SwapInArgs, stream=None) -> None:
    """Launch hs_swap_in with a prepared argument block."""
    _capi.check(_lib().hs_swap_in(C.byref(args), C.c_void_p(_stream(stream))), "hs_swap_in")


def swap_in_timeout_selftest(args: SwapInArgs, *, rank=-1, which=0, stream=None) -> None:
    """hs_swap_in with one CTA of every full-path row giving up a bounded wait at
    once (``rank`` of the row's cluster, the last when negative; ``which`` 0 =
    the staged-state wait, 1 = the top-k-row wait): those rows must report
    exactly HS_ST_TIMEOUT and write nothing else."""
    _capi.check(_lib().hs_swap_in_timeout_selftest(C.byref(args), int(rank), int(which),
                                                   C.c_void_p(_stream(stream))),
                "hs_swap_in_timeout_selftest")


def layer_args_array(layers):
    """A ctypes array of hs_swap_in_args from a list of ``make_swap_in_args``
    results (one per layer); keeps the layers' tensors alive with it."""
    arr = (SwapInArgs * len(layers))(*layers)
    arr.keep = list(layers)
    return arr


def swap_in_layers(layers, stream=None) -> None:
    """hs_swap_in_layers: every layer's swap-in in one launch.  ``layers`` is a
    list of ``make_swap_in_args`` results (same geometry, other pointers) or an
    array from ``layer_args_array`` (cheaper to reuse)."""
    arr = layers if isinstance(layers, C.Array) else layer_args_array(layers)
    _capi.check(_lib().hs_swap_in_layers(arr, len(arr), C.c_void_p(_stream(stream))),
                "hs_swap_in_layers")


def swap_in_layers_timeout_selftest(layers, *, which=0, stream=None) -> None:
    """hs_swap_in_layers with every full-path row giving up one bounded wait at
    once (``which`` 0 = the staged state, 1 = the top-k row)."""
    arr = layers if isinstance(layers, C.Array) else layer_args_array(layers)
    _capi.check(_lib().hs_swap_in_layers_timeout_selftest(arr, len(arr), int(which),
                                                          C.c_void_p(_stream(stream))),
                "hs_swap_in_layers_timeout_selftest")


def swap_in(*, stream=None, **tensors) -> None:
    """One swap-in call; keyword tensors as in ``make_swap_in_args``."""
    swap_in_args(make_swap_in_args(**tensors), stream)


def invalidate_tokens(slot_tokens, state_rows, tokens, *, hot_size=None, status=None,
                      stream=None) -> None:
    """Slots [0, hot_size) of state row state_rows[n] that hold token tokens[n] become -1."""
    _need(slot_tokens, torch.int32, "slot_tokens", 2)
    _need(state_rows, torch.int64, "state_rows", 1)
    _need(tokens, torch.int32, "tokens", 1)
    if state_rows.numel() != tokens.numel():
        raise ValueError("state_rows and tokens differ in length")
    H = int(hot_size if hot_size is not None else slot_tokens.shape[1] - 1)
    _capi.check(_lib().hs_invalidate_tokens(
        _ptr(slot_tokens), slot_tokens.stride(0), H, slot_tokens.shape[0], _ptr(state_rows),
        _ptr(tokens), tokens.numel(), _ptr(status), C.c_void_p(_stream(stream))),
        "hs_invalidate_tokens")


def wait_selftest(max_polls, status, *, stream=None) -> None:
    """Run the bounded mbarrier wait on a barrier that nothing arms (at most
    max_polls polls); HS_ST_TIMEOUT is OR-ed into ``status`` (int32 [1])."""
    _need(status, torch.int32, "status", 1)
    _capi.check(_lib().hs_wait_selftest(int(max_polls), _ptr(status),
                                        C.c_void_p(_stream(stream))), "hs_wait_selftest")


def gather_misses(pool_layers, hot_layers, miss_src, miss_dst, miss_count, *, has_v=False,
                  status=None, stream=None, ptrs=None, overlap_prev=False) -> None:
    """Replay a swap-in's miss plan onto layers that share its indices: in every
    layer, hot row miss_dst[b][m] = pool row miss_src[b][m] for m < miss_count[b].
    ``pool_layers`` / ``hot_layers`` are lists of per-layer tensors [rows, ...]
    (K layers, then V layers when has_v); ``ptrs`` may pass prebuilt pointer
    arrays (pool_ptrs, hot_ptrs) from ``layer_pointer_array``; pass them when
    capturing a CUDA graph (building them copies to the device).  With
    ``overlap_prev`` the launch may start while the preceding kernel in the
    stream still runs; it reads the plan only once that kernel has finished."""
    _need(miss_src, torch.int64, "miss_src", 2)
    _need(miss_dst, torch.int32, "miss_dst", 2)
    _need(miss_count, torch.int32, "miss_count", 1)
    if miss_src.stride(0) != miss_dst.stride(0) or miss_src.shape != miss_dst.shape:
        raise ValueError("miss_src and miss_dst need the same shape and row stride")
    if len(pool_layers) != len(hot_layers) or not pool_layers:
        raise ValueError("need matching non-empty layer lists")
    if has_v and len(pool_layers) % 2:
        raise ValueError("with has_v the lists hold K layers then V layers")
    B, K = miss_src.shape
    if miss_count.numel() < B:
        raise ValueError("miss_count needs one entry per batch row")
    geo_p = {_byte_rows(t, "pool")[2:] for t in pool_layers}
    geo_h = {_byte_rows(t, "hot")[2:] for t in hot_layers}
    if len(geo_p) != 1 or len(geo_h) != 1 or geo_p != geo_h or len({*geo_p.pop()}) != 1:
        raise ValueError("every pool and hot layer needs contiguous rows of one byte width")
    rb = _byte_rows(pool_layers[0], "pool")[2]
    if ptrs is None:
        dev = miss_src.device
        ptrs = (layer_pointer_array(pool_layers, dev), layer_pointer_array(hot_layers, dev))
    nl = len(pool_layers) // (2 if has_v else 1)
    _capi.check(_lib().hs_gather_misses(
        _ptr(ptrs[0]), _ptr(ptrs[1]), nl,
        (1 if has_v else 0) | (_capi.OVERLAP_PREV if overlap_prev else 0),
        min(t.shape[0] for t in pool_layers), min(t.shape[0] for t in hot_layers), rb,
        _ptr(miss_src), _ptr(miss_dst), miss_src.stride(0), _ptr(miss_count), B, K,
        _ptr(status), C.c_void_p(_stream(stream))), "hs_gather_misses")


_FP8_IN = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}


def fp8_store_kv(k, v, k_cache, v_cache, cache_loc, *, k_scale=None, v_scale=None,
                 page_size=16, status=None, stream=None) -> None:
    """Quantise K/V [T, heads, dim] (or [T, heads*dim]) to FP8 E4M3 and scatter token t
    to slot cache_loc[t] of a paged cache ([pages, page_size, heads, dim] or
    [slots, heads, dim]; uint8 or float8_e4m3fn).  With k_scale and v_scale
    (device fp32 tensors of one element) values are multiplied by fp32(1/scale)."""
    _need(cache_loc, torch.int64, "cache_loc", 1)
    if k.dtype not in _FP8_IN or (v is not None and v.dtype != k.dtype):
        raise TypeError("k and v must both be float32, float16 or bfloat16")
    if (v is None) != (v_cache is None):
        raise ValueError("v and v_cache go together")
    if k_cache.element_size() != 1 or (v_cache is not None and v_cache.element_size() != 1):
        raise TypeError("caches must be 1-byte tensors (uint8 or float8_e4m3fn)")
    if k_cache.dim() == 4:
        _, ps, heads, dim = k_cache.shape
        if ps != page_size:
            raise ValueError(f"page_size mismatch: cache has {ps}, expected {page_size}")
        c_page, c_off, c_head = k_cache.stride(0), k_cache.stride(1), k_cache.stride(2)
        num_slots = k_cache.shape[0] * ps
    elif k_cache.dim() == 3:
        _, heads, dim = k_cache.shape
        c_page, c_off, c_head = k_cache.stride(0) * page_size, k_cache.stride(0), k_cache.stride(1)
        num_slots = k_cache.shape[0] // page_size * page_size
    else:
        raise ValueError("caches must be 3-D or 4-D")
    if k_cache.stride(-1) != 1 or (v_cache is not None and v_cache.stride() != k_cache.stride()):
        raise ValueError("caches need contiguous dims and the same layout")
    T = k.shape[0]
    if k.dim() == 2:
        k = k.view(T, heads, dim)
        v = v.view(T, heads, dim) if v is not None else None
    for t, name in ((k, "k"), (v, "v")):
        if t is not None and (tuple(t.shape) != (T, heads, dim) or t.stride(2) != 1):
            raise ValueError(f"{name} must be [T, {heads}, {dim}] with a contiguous last dim")
    if cache_loc.numel() != T:
        raise ValueError("cache_loc needs one entry per token")
    for sc, name in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        if sc is not None:
            _need(sc, torch.float32, name)
    _capi.check(_lib().hs_fp8_store_kv(
        _ptr(k), _ptr(v), _FP8_IN[k.dtype], k.stride(0), k.stride(1),
        v.stride(0) if v is not None else 0, v.stride(1) if v is not None else 0,
        _ptr(k_cache), _ptr(v_cache), c_page, c_off, c_head, page_size, num_slots,
        _ptr(cache_loc), T, heads, dim, _ptr(k_scale), _ptr(v_scale), _ptr(status),
        C.c_void_p(_stream(stream))), "hs_fp8_store_kv")


def store_kv(k_src, v_src, k_dst, v_dst, loc, status=None, stream=None) -> None:
    """k_dst[loc[t]] = k_src[t] and v_dst[loc[t]] = v_src[t] (v_* may be None)."""
    _need(loc, torch.int64, "loc", 1)
    ks, n, rb, ksp = _byte_rows(k_src, "k_src")
    kd, drows, rbd, dp = _byte_rows(k_dst, "k_dst")
    if rbd != rb:
        raise ValueError("k_src and k_dst rows differ in width")
    vs = vd = None
    vsp = 0
    if v_src is not None or v_dst is not None:
        if v_src is None or v_dst is None:
            raise ValueError("v_src and v_dst go together")
        vs, vn, vrb, vsp = _byte_rows(v_src, "v_src")
        vd, vdrows, vdrb, vdp = _byte_rows(v_dst, "v_dst")
        if vn != n or vrb != rb or vdrb != rb or vdp != dp:
            raise ValueError("V tensors must match K in rows, width and destination pitch")
        drows = min(drows, vdrows)
    if loc.numel() != n:
        raise ValueError("loc needs one entry per source row")
    _capi.check(_lib().hs_store_kv(ks, vs, ksp, vsp, kd, vd, dp, drows, _ptr(loc), n, rb,
                                   _ptr(status), C.c_void_p(_stream(stream))), "hs_store_kv")


def transfer_kv(src_ptrs, dst_ptrs, src_idx, dst_idx, *, num_layers, has_v, src_stride,
                dst_stride, src_rows, dst_rows, row_bytes, status=None, stream=None,
                device_sources=False) -> None:
    """Raw hs_transfer_kv: device uint64 pointer arrays and int64 index arrays;
    ``device_sources`` asserts every source is device memory (bulk copies)."""
    _need(src_idx, torch.int64, "src_idx", 1)
    _need(dst_idx, torch.int64, "dst_idx", 1)
    if src_idx.numel() != dst_idx.numel():
        raise ValueError("src_idx and dst_idx differ in length")
    _capi.check(_lib().hs_transfer_kv(
        _ptr(src_ptrs), _ptr(dst_ptrs), num_layers,
        int(bool(has_v)) | (_capi.XFER_DEVICE_SOURCES if device_sources else 0), _ptr(src_idx),
        _ptr(dst_idx), src_idx.numel(), src_stride, dst_stride, src_rows, dst_rows, row_bytes,
        _ptr(status), C.c_void_p(_stream(stream))), "hs_transfer_kv")


def layer_pointer_array(layers, device) -> torch.Tensor:
    """Device uint64-as-int64 array of the layers' base addresses."""
    return torch.tensor([int(t.data_ptr()) for t in layers], dtype=torch.int64, device=device)


def transfer_kv_layers(src_layers, dst_layers, src_idx, dst_idx, *, has_v=False, status=None,
                       stream=None, ptrs=None) -> None:
    """Convenience form over lists of per-layer tensors [rows, ...] (K layers then V
    layers when has_v).  ``ptrs`` may pass prebuilt (src_ptrs, dst_ptrs)."""
    if len(src_layers) != len(dst_layers) or not src_layers:
        raise ValueError("need matching non-empty layer lists")
    geo_s = {_byte_rows(t, "src")[2:] for t in src_layers}
    geo_d = {_byte_rows(t, "dst")[2:] for t in dst_layers}
    if len(geo_s) != 1 or len(geo_d) != 1:
        raise ValueError("all layers need the same row width and pitch")
    (rb, sp), (rbd, dp) = geo_s.pop(), geo_d.pop()
    if rb != rbd:
        raise ValueError("source and destination rows differ in width")
    nl = len(src_layers) // (2 if has_v else 1)
    if ptrs is None:
        dev = src_idx.device
        ptrs = (layer_pointer_array(src_layers, dev), layer_pointer_array(dst_layers, dev))
    transfer_kv(ptrs[0], ptrs[1], src_idx, dst_idx, num_layers=nl, has_v=has_v, src_stride=sp,
                dst_stride=dp, src_rows=min(t.shape[0] for t in src_layers),
                dst_rows=min(t.shape[0] for t in dst_layers), row_bytes=rb, status=status,
                stream=stream, device_sources=all(t.is_cuda for t in src_layers))


def probe_read(src, sink, stream=None) -> None:
    """Stream-read every byte of ``src`` (device or pinned host) into ``sink``."""
    ptr, n, rb, pitch = _byte_rows(src.view(-1), "src")
    _capi.check(_lib().hs_probe_read(ptr, n * rb, _ptr(sink), C.c_void_p(_stream(stream))),
                "hs_probe_read")
