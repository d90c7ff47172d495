"""The C-ABI library builds, loads without a GPU, exports exactly what
include/hisparse.h declares, and rejects bad arguments synchronously before
touching the GPU."""
from __future__ import annotations

import ctypes as C
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from sparse_attention_kv_row_gb300 import _capi, build

    build.build()
    return _capi.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "hisparse.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"\b(hs_[a-z0-9_]+)\s*\(", src))


def test_exports_match_header(lib):
    from sparse_attention_kv_row_gb300 import _capi

    declared = _declared()
    assert declared == set(_capi.EXPORTS)
    out = subprocess.run(["nm", "-D", "--defined-only", _capi.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (hs_[a-z0-9_]+)$", out, flags=re.M))
    assert declared <= exported, declared - exported
    assert lib.hs_abi_version() == _capi.ABI_VERSION


def test_error_strings(lib):
    assert lib.hs_err_string(0) == b"HS_OK"
    assert b"ARG" in lib.hs_err_string(1)
    for bit, name in ((1, b"HS_ST_DUP_ID"), (2, b"HS_ST_BAD_POOL_ROW"), (4, b"HS_ST_BAD_LRU_SLOT"),
                      (8, b"HS_ST_BAD_HOT_ROW"), (16, b"HS_ST_TIMEOUT"), (32, b"HS_ST_BAD_STATE"),
                      (64, b"HS_ST_BAD_INDEX")):
        assert lib.hs_status_string(bit) == name
    assert lib.hs_status_string(3) == b""


def _args(**kw):
    from sparse_attention_kv_row_gb300 import SwapInArgs

    base = dict(batch=2, top_k=4, hot_size=8, flags=0, row_bytes=16, topk_stride=4,
                out_stride=4, slot_tokens_stride=9, slot_rows_stride=9, lru_stride=8,
                pool_rows_cols=10, pool_rows_stride=10, num_states=2, pool_num_rows=20,
                hot_num_rows=18)
    base.update(kw)
    return SwapInArgs(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(top_k=9), 2),             # top_k > hot_size
    (dict(hot_size=0), 2),
    (dict(hot_size=40000, top_k=4), 2),
    (dict(batch=-1), 1),
    (dict(row_bytes=0), 1),
    (dict(flags=8), 1),
    (dict(flags=16), 1),
    (dict(), 1),                    # required pointers are NULL
])
def test_swap_in_rejects(lib, kw, code):
    rc = lib.hs_swap_in(C.byref(_args(**kw)), None)
    assert rc == code
    assert lib.hs_last_error() != b""


def test_swap_in_null_args(lib):
    assert lib.hs_swap_in(None, None) == 1


def test_empty_work_is_ok_without_gpu(lib):
    assert lib.hs_swap_in(C.byref(_args(batch=0)), None) == 0
    assert lib.hs_swap_in(C.byref(_args(top_k=0)), None) == 0
    assert lib.hs_store_kv(None, None, 16, 16, None, None, 16, 10, None, 0, 16, None, None) == 0
    assert lib.hs_transfer_kv(None, None, 3, 0, None, None, 0, 16, 16, 1, 1, 16, None, None) == 0


def test_plan_arguments_rejected(lib):
    """The miss-plan arguments are checked before any device call."""
    a = _args()
    for k in ("topk_ids", "seq_lens", "req_state", "slot_tokens", "slot_rows", "lru",
              "pool_rows", "pool_k", "hot_k", "out_rows"):
        setattr(a, k, 256)  # never dereferenced: the checks below fail first
    a.miss_src = 512
    assert lib.hs_swap_in(C.byref(a), None) == 1   # miss_src without miss_dst
    assert b"miss_dst" in lib.hs_last_error()
    a.miss_dst = 768
    assert lib.hs_swap_in(C.byref(a), None) == 1   # plan without miss_count
    a.miss_count, a.plan_stride = 1024, 2
    assert lib.hs_swap_in(C.byref(a), None) == 1   # plan_stride < top_k
    a.miss_src = a.miss_dst = None
    a.miss_mask, a.mask_stride = 512, 3
    assert lib.hs_swap_in(C.byref(a), None) == 1   # mask_stride < top_k
    assert b"mask_stride" in lib.hs_last_error()


def test_gather_rejects(lib):
    g = lib.hs_gather_misses
    assert g(None, None, 3, 0, 10, 10, 16, None, None, 4, None, 0, 4, None, None) == 0  # no rows
    assert g(None, None, 0, 0, 10, 10, 16, None, None, 4, None, 2, 4, None, None) == 0  # no layers
    assert g(None, None, 3, 0, 10, 10, 16, None, None, 4, None, 2, 4, None, None) == 1  # NULLs
    assert g(8, 8, 3, 0, 10, 10, 16, 8, 8, 2, 8, 2, 4, None, None) == 1  # plan_stride < top_k
    assert g(8, 8, 3, 2, 10, 10, 16, 8, 8, 4, 8, 2, 4, None, None) == 1  # unknown flag bit
    assert g(8, 8, 3, 0, 10, 10, 0, 8, 8, 4, 8, 2, 4, None, None) == 1  # row_bytes < 1


def test_movers_reject(lib):
    assert lib.hs_store_kv(None, None, 16, 16, None, None, 16, 10, None, 5, 16, None, None) == 1
    assert lib.hs_store_kv(1, None, 8, 0, 1, None, 16, 10, 1, 5, 16, None, None) == 1  # stride
    assert lib.hs_store_kv(1, 1, 16, 16, 1, None, 16, 10, 1, 5, 16, None, None) == 1  # v pair
    assert lib.hs_transfer_kv(1, 1, 3, 4, 1, 1, 5, 16, 16, 1, 1, 16, None, None) == 1  # flags
    assert lib.hs_transfer_kv(1, 1, 3, 0, 1, 1, 5, 8, 16, 1, 1, 16, None, None) == 1  # stride
    assert lib.hs_probe_read(8, 32, 16, None) == 1  # misaligned source
    assert lib.hs_wait_selftest(-1, 8, None) == 1   # negative poll budget
    assert lib.hs_wait_selftest(10, None, None) == 1  # no status word


def test_smem_bytes(lib):
    assert lib.hs_swap_in_smem_bytes(2048, 4096) > 0
    assert lib.hs_swap_in_smem_bytes(4097, 4096) == 0
    assert lib.hs_swap_in_smem_bytes(1, 32768) == 0
    assert lib.hs_swap_in_smem_bytes(2048, 4096) < 227 * 1024


def test_nvtx_ranges_switch_on_without_a_profiler():
    """HS_NVTX=1 wraps each call in an NVTX range; with no profiler attached the
    calls behave exactly as without it (here: argument errors, no GPU needed)."""
    import subprocess
    import sys

    code = ("import ctypes, sys; sys.path.insert(0, '.'); "
            "from sparse_attention_kv_row_gb300 import _capi; lib = _capi.load(); "
            "assert lib.hs_swap_in(None, None) == 1; "
            "assert lib.hs_store_kv(None, None, 16, 16, None, None, 16, 10, None, 5, 16, None, None) == 1; "
            "assert lib.hs_swap_in_layers(None, 1, None) == 1; print('ok')")
    env = dict(os.environ, HS_NVTX="1")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stderr
