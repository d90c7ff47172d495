"""Pins for the oracle's indexed row movers against numpy advanced-index
assignment (a library routine), as the pages define them:
tokenspeed tokenspeed_kernel/ops/kvcache/triton.py, store_kv_cache
("k_dst[loc] = k_src; v_dst[loc] = v_src") and transfer_kv_per_layer /
transfer_kv_all_layer (per layer: dst[dst_idx] = src[src_idx])."""
from __future__ import annotations

import numpy as np
import pytest

import oracle


@pytest.mark.parametrize("S", [1, 3, 4, 132, 656, 2048])
def test_store_kv_matches_index_assignment(S):
    rng = np.random.default_rng(S)
    n, rows = 37, 211
    k_src = rng.integers(0, 256, (n, S), dtype=np.uint8)
    v_src = rng.integers(0, 256, (n, S), dtype=np.uint8)
    k_dst = rng.integers(0, 256, (rows, S), dtype=np.uint8)
    v_dst = rng.integers(0, 256, (rows, S), dtype=np.uint8)
    loc = rng.choice(rows, size=n, replace=False).astype(np.int64)
    ek, ev = k_dst.copy(), v_dst.copy()
    ek[loc] = k_src
    ev[loc] = v_src
    st = np.zeros(1, np.int32)
    oracle.store_kv(k_src=k_src, v_src=v_src, k_dst=k_dst, v_dst=v_dst, loc=loc, status=st)
    np.testing.assert_array_equal(k_dst, ek)
    np.testing.assert_array_equal(v_dst, ev)
    assert st[0] == 0


def test_store_kv_strided_source_and_bad_index():
    rng = np.random.default_rng(1)
    S, n, rows = 24, 10, 50
    qkv = rng.integers(0, 256, (n, 3 * S), dtype=np.uint8)  # split view: stride 3S
    k_src, v_src = qkv[:, S:2 * S], qkv[:, 2 * S:]
    k_dst = np.zeros((rows, S), np.uint8)
    v_dst = np.zeros((rows, S), np.uint8)
    loc = rng.choice(rows, size=n, replace=False).astype(np.int64)
    loc[3] = rows  # out of range: skipped, status bit
    loc[7] = -2
    ek, ev = k_dst.copy(), v_dst.copy()
    ok = (loc >= 0) & (loc < rows)
    ek[loc[ok]] = k_src[ok]
    ev[loc[ok]] = v_src[ok]
    st = np.zeros(1, np.int32)
    oracle.store_kv(k_src=k_src, v_src=v_src, k_dst=k_dst, v_dst=v_dst, loc=loc, status=st)
    np.testing.assert_array_equal(k_dst, ek)
    np.testing.assert_array_equal(v_dst, ev)
    assert st[0] == oracle.ST_BAD_INDEX


def test_store_kv_k_only():
    rng = np.random.default_rng(2)
    k_src = rng.integers(0, 256, (5, 7), dtype=np.uint8)
    k_dst = np.zeros((9, 7), np.uint8)
    loc = np.array([8, 0, 4, 2, 6], np.int64)
    e = k_dst.copy()
    e[loc] = k_src
    oracle.store_kv(k_src=k_src, v_src=None, k_dst=k_dst, v_dst=None, loc=loc)
    np.testing.assert_array_equal(k_dst, e)


@pytest.mark.parametrize("L,S", [(1, 656), (3, 132), (5, 4), (2, 1)])
def test_transfer_matches_index_assignment(L, S):
    rng = np.random.default_rng(L * 1000 + S)
    n, src_rows, dst_rows = 53, 300, 120
    src = [rng.integers(0, 256, (src_rows, S), dtype=np.uint8) for _ in range(L)]
    dst = [rng.integers(0, 256, (dst_rows, S), dtype=np.uint8) for _ in range(L)]
    src_idx = rng.integers(0, src_rows, n).astype(np.int64)  # repeats allowed
    dst_idx = rng.choice(dst_rows, size=n, replace=False).astype(np.int64)
    exp = [d.copy() for d in dst]
    for e, s in zip(exp, src):
        e[dst_idx] = s[src_idx]
    oracle.transfer_kv(src_layers=src, dst_layers=dst, src_idx=src_idx, dst_idx=dst_idx)
    for d, e in zip(dst, exp):
        np.testing.assert_array_equal(d, e)


def test_transfer_bad_index_skips_pair():
    rng = np.random.default_rng(9)
    S = 16
    src = [rng.integers(0, 256, (10, S), dtype=np.uint8) for _ in range(2)]
    dst = [np.zeros((6, S), np.uint8) for _ in range(2)]
    src_idx = np.array([0, 10, 3, -1], np.int64)
    dst_idx = np.array([5, 1, 6, 2], np.int64)
    st = np.zeros(1, np.int32)
    oracle.transfer_kv(src_layers=src, dst_layers=dst, src_idx=src_idx, dst_idx=dst_idx,
                       status=st)
    for l in range(2):
        e = np.zeros((6, S), np.uint8)
        e[5] = src[l][0]
        np.testing.assert_array_equal(dst[l], e)
    assert st[0] == oracle.ST_BAD_INDEX
