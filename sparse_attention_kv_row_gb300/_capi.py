"""ctypes declarations of libhisparse's C ABI (include/hisparse.h).

Loading never falls back to anything: if the shared library is missing or
does not export the full ABI, ``load()`` raises.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libhisparse.so")

HS_OK, HS_ERR_ARG, HS_ERR_UNSUPPORTED, HS_ERR_CUDA = 0, 1, 2, 3
ST_DUP_ID = 1
ST_BAD_POOL_ROW = 2
ST_BAD_LRU_SLOT = 4
ST_BAD_HOT_ROW = 8
ST_TIMEOUT = 16
ST_BAD_STATE = 32
ST_BAD_INDEX = 64
SEQ_LENS_I64 = 1
REQ_STATE_I64 = 2
OVERLAP_PREV = 4
DT_F32, DT_F16, DT_BF16 = 0, 1, 2
XFER_HAS_V, XFER_DEVICE_SOURCES = 1, 2
ABI_VERSION = 8

# Every symbol include/hisparse.h declares.
EXPORTS = ("hs_swap_in", "hs_swap_in_smem_bytes", "hs_store_kv", "hs_transfer_kv",
           "hs_gather_misses", "hs_fp8_store_kv", "hs_invalidate_tokens", "hs_probe_read", "hs_err_string", "hs_status_string", "hs_last_error",
           "hs_abi_version", "hs_wait_selftest", "hs_swap_in_timeout_selftest",
           "hs_swap_in_layers", "hs_swap_in_layers_timeout_selftest")


class SwapInArgs(C.Structure):
    """Mirror of ``hs_swap_in_args``."""
    _fields_ = [
        ("batch", C.c_int32), ("top_k", C.c_int32), ("hot_size", C.c_int32),
        ("flags", C.c_int32),
        ("num_real", C.c_void_p),
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


class HisparseError(RuntimeError):
    def __init__(self, code: int, where: str, msg: str):
        super().__init__(f"{where}: {msg} (hs_err {code})")
        self.code = code


_lock = threading.Lock()
_lib: C.CDLL | None = None


def load() -> C.CDLL:
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"libhisparse.so is not built ({LIB_PATH}); run "
                "`python -m sparse_attention_kv_row_gb300.build` (needs nvcc). "
                "There is no fallback implementation.")
        lib = C.CDLL(LIB_PATH)
        missing = [s for s in EXPORTS if not hasattr(lib, s)]
        if missing:
            raise ImportError(f"libhisparse.so lacks exports: {missing}")
        vp, i32, i64 = C.c_void_p, C.c_int32, C.c_int64
        lib.hs_swap_in.argtypes = [C.POINTER(SwapInArgs), vp]
        lib.hs_swap_in.restype = C.c_int
        lib.hs_swap_in_timeout_selftest.argtypes = [C.POINTER(SwapInArgs), i32, i32, vp]
        lib.hs_swap_in_timeout_selftest.restype = C.c_int
        lib.hs_swap_in_layers.argtypes = [C.POINTER(SwapInArgs), i32, vp]
        lib.hs_swap_in_layers.restype = C.c_int
        lib.hs_swap_in_layers_timeout_selftest.argtypes = [C.POINTER(SwapInArgs), i32, i32, vp]
        lib.hs_swap_in_layers_timeout_selftest.restype = C.c_int
        lib.hs_swap_in_smem_bytes.argtypes = [i32, i32]
        lib.hs_swap_in_smem_bytes.restype = i64
        lib.hs_store_kv.argtypes = [vp, vp, i64, i64, vp, vp, i64, i64, vp, i64, i64, vp, vp]
        lib.hs_store_kv.restype = C.c_int
        lib.hs_transfer_kv.argtypes = [vp, vp, i32, i32, vp, vp, i64, i64, i64, i64, i64, i64,
                                       vp, vp]
        lib.hs_transfer_kv.restype = C.c_int
        lib.hs_gather_misses.argtypes = [vp, vp, i32, i32, i64, i64, i64, vp, vp, i64, vp, i32,
                                         i32, vp, vp]
        lib.hs_gather_misses.restype = C.c_int
        lib.hs_fp8_store_kv.argtypes = [vp, vp, i32, i64, i64, i64, i64, vp, vp, i64, i64, i64,
                                        i32, i64, vp, i64, i32, i32, vp, vp, vp, vp]
        lib.hs_fp8_store_kv.restype = C.c_int
        lib.hs_invalidate_tokens.argtypes = [vp, i64, i32, i64, vp, vp, i64, vp, vp]
        lib.hs_invalidate_tokens.restype = C.c_int
        lib.hs_probe_read.argtypes = [vp, i64, vp, vp]
        lib.hs_probe_read.restype = C.c_int
        lib.hs_err_string.argtypes = [i32]
        lib.hs_err_string.restype = C.c_char_p
        lib.hs_status_string.argtypes = [i32]
        lib.hs_status_string.restype = C.c_char_p
        lib.hs_last_error.argtypes = []
        lib.hs_last_error.restype = C.c_char_p
        lib.hs_wait_selftest.argtypes = [i32, vp, vp]
        lib.hs_wait_selftest.restype = i32
        lib.hs_abi_version.argtypes = []
        lib.hs_abi_version.restype = i32
        if lib.hs_abi_version() != ABI_VERSION:
            raise ImportError("libhisparse.so ABI version mismatch; rebuild it")
        _lib = lib
        return lib


def check(code: int, where: str) -> None:
    if code != HS_OK:
        lib = load()
        raise HisparseError(code, where, lib.hs_last_error().decode(errors="replace"))
