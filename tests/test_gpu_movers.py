"""GPU parity for hs_store_kv and hs_transfer_kv against the CPU oracle,
element by element, through the C ABI: every copy width (16-byte, 4-byte,
byte), strided sources, K-only and K+V, per-layer and all-layer, pinned-host
sources, out-of-range indices and empty calls."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__

    __graft_entry__.build()
    return torch.device("cuda:0")


def _hs():
    import sparse_attention_kv_row_gb300 as hs

    return hs


# 16-byte rows up to 2048 B take the form that loads a row with its slot
# index (U = 1, 2 or 4 chunks per lane; 400 and 656 B leave some lanes a
# chunk short), longer or unaligned rows the general one.
@pytest.mark.parametrize("S,n,rows,with_v", [(2048, 4096, 9000, True), (656, 333, 1000, False),
                                              (400, 900, 2000, True), (512, 700, 1600, False),
                                              (4096, 300, 1000, True),
                                              (132, 1000, 5000, True), (17, 77, 300, True),
                                              (4, 3000, 3001, False)])
def test_store_kv_parity(dev, S, n, rows, with_v):
    rng = np.random.default_rng(S + n)
    k_src = rng.integers(0, 256, (n, S), dtype=np.uint8)
    v_src = rng.integers(0, 256, (n, S), dtype=np.uint8) if with_v else None
    k_dst = rng.integers(0, 256, (rows, S), dtype=np.uint8)
    v_dst = rng.integers(0, 256, (rows, S), dtype=np.uint8) if with_v else None
    loc = rng.choice(rows, size=n, replace=False).astype(np.int64)
    loc[rng.integers(n, size=3)] = [rows, -1, rows + 100]
    g = {k: (torch.from_numpy(v.copy()).to(dev) if v is not None else None)
         for k, v in dict(k_src=k_src, v_src=v_src, k_dst=k_dst, v_dst=v_dst, loc=loc).items()}
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    _hs().store_kv(g["k_src"], g["v_src"], g["k_dst"], g["v_dst"], g["loc"], status=st)
    r_st = np.zeros(1, np.int32)
    oracle.store_kv(k_src=k_src, v_src=v_src, k_dst=k_dst, v_dst=v_dst, loc=loc, status=r_st)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(g["k_dst"].cpu().numpy(), k_dst)
    if with_v:
        np.testing.assert_array_equal(g["v_dst"].cpu().numpy(), v_dst)
    assert st.item() == r_st[0] == oracle.ST_BAD_INDEX


def test_store_kv_strided_bf16_source(dev):
    """Sources as views of a fused qkv tensor (leading stride > row), bf16 rows."""
    rng = np.random.default_rng(1)
    n, heads, hd, rows = 257, 8, 128, 4000
    qkv = torch.from_numpy(rng.standard_normal((n, 3, heads, hd)).astype(np.float32)).to(
        torch.bfloat16)
    k_src, v_src = qkv[:, 1], qkv[:, 2]
    k_dst = torch.zeros((rows, heads, hd), dtype=torch.bfloat16)
    v_dst = torch.zeros((rows, heads, hd), dtype=torch.bfloat16)
    loc = torch.from_numpy(rng.choice(rows, size=n, replace=False).astype(np.int64))
    gk, gv = k_dst.to(dev), v_dst.to(dev)
    _hs().store_kv(k_src.to(dev), v_src.to(dev), gk, gv, loc.to(dev))
    k_dst[loc] = k_src
    v_dst[loc] = v_src
    torch.cuda.synchronize()
    assert torch.equal(gk.cpu().view(torch.int16), k_dst.view(torch.int16))
    assert torch.equal(gv.cpu().view(torch.int16), v_dst.view(torch.int16))


@pytest.mark.parametrize("L,S,has_v,host", [(61, 656, False, True), (1, 656, True, False),
                                             (4, 132, False, True), (3, 9, True, False),
                                             (2, 2048, True, True)])
def test_transfer_parity(dev, L, S, has_v, host):
    rng = np.random.default_rng(L * 31 + S)
    n, src_rows, dst_rows = 1500, 6000, 2000
    P = L * (2 if has_v else 1)
    src = [rng.integers(0, 256, (src_rows, S), dtype=np.uint8) for _ in range(P)]
    dst = [rng.integers(0, 256, (dst_rows, S), dtype=np.uint8) for _ in range(P)]
    src_idx = rng.integers(0, src_rows, n).astype(np.int64)
    dst_idx = rng.choice(dst_rows, size=n, replace=False).astype(np.int64)
    src_idx[5], dst_idx[9] = src_rows, -3  # two bad pairs
    g_src = [torch.from_numpy(x.copy()).pin_memory() if host else torch.from_numpy(x).to(dev)
             for x in src]
    g_dst = [torch.from_numpy(x.copy()).to(dev) for x in dst]
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    _hs().transfer_kv_layers(g_src, g_dst, torch.from_numpy(src_idx).to(dev),
                             torch.from_numpy(dst_idx).to(dev), has_v=has_v, status=st)
    r_st = np.zeros(1, np.int32)
    oracle.transfer_kv(src_layers=src, dst_layers=dst, src_idx=src_idx, dst_idx=dst_idx,
                       status=r_st)
    torch.cuda.synchronize()
    for l in range(P):
        np.testing.assert_array_equal(g_dst[l].cpu().numpy(), dst[l], err_msg=f"layer {l}")
    assert st.item() == r_st[0] == oracle.ST_BAD_INDEX


@pytest.mark.parametrize("offset", [0, 4, 1])
def test_transfer_bulk_path_with_layer_bases_off_16_bytes(dev, offset):
    """Device sources with 16-byte row pitches take the bulk (TMA) path; a layer
    whose base address is off 16 bytes (views 4 or 1 bytes into a buffer) is
    copied row by row in words or bytes instead.  Same results as the oracle."""
    rng = np.random.default_rng(40 + offset)
    L, S, n, src_rows, dst_rows = 3, 656, 2000, 5000, 2500
    src = [rng.integers(0, 256, (src_rows, S), dtype=np.uint8) for _ in range(L)]
    dst = [rng.integers(0, 256, (dst_rows, S), dtype=np.uint8) for _ in range(L)]
    src_idx = rng.integers(0, src_rows, n).astype(np.int64)
    dst_idx = rng.choice(dst_rows, size=n, replace=False).astype(np.int64)
    g_src = []
    for l, x in enumerate(src):
        off = offset if l == 1 else 0   # only the middle layer is off 16 bytes
        buf = torch.zeros(src_rows * S + 16, dtype=torch.uint8, device=dev)
        view = buf[off: off + src_rows * S].view(src_rows, S)
        view.copy_(torch.from_numpy(x))
        g_src.append(view)
    g_dst = [torch.from_numpy(x.copy()).to(dev) for x in dst]
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    _hs().transfer_kv_layers(g_src, g_dst, torch.from_numpy(src_idx).to(dev),
                             torch.from_numpy(dst_idx).to(dev), status=st)
    r_st = np.zeros(1, np.int32)
    oracle.transfer_kv(src_layers=src, dst_layers=dst, src_idx=src_idx, dst_idx=dst_idx,
                       status=r_st)
    torch.cuda.synchronize()
    for l in range(L):
        np.testing.assert_array_equal(g_dst[l].cpu().numpy(), dst[l], err_msg=f"layer {l}")
    assert st.item() == r_st[0] == 0


def test_empty_calls_launch_nothing(dev):
    hs = _hs()
    z = torch.zeros((0, 16), dtype=torch.uint8, device=dev)
    loc = torch.zeros(0, dtype=torch.int64, device=dev)
    hs.store_kv(z, None, torch.zeros((4, 16), dtype=torch.uint8, device=dev), None, loc)
    src = [torch.zeros((4, 16), dtype=torch.uint8, device=dev)]
    hs.transfer_kv_layers(src, src, loc, loc)


def test_probe_read(dev):
    hs = _hs()
    buf = torch.arange(1 << 20, dtype=torch.int32).pin_memory()
    sink = torch.zeros(1, dtype=torch.int64, device=dev)
    hs.probe_read(buf, sink)
    torch.cuda.synchronize()
    x = np.bitwise_xor.reduce(np.arange(1 << 20, dtype=np.uint32))
    assert (sink.item() & 0xFFFFFFFF) == int(x)


@pytest.mark.parametrize("n", [1, 2, 7])
def test_transfer_bulk_path_few_pairs_many_layers(dev, n):
    """The bulk path runs its units layer-major (u = pointer pair * n + pair);
    with one pair the divisor is 1.  K and V of five layers, device sources."""
    rng = np.random.default_rng(70 + n)
    L, S, src_rows, dst_rows = 5, 656, 50, 40
    P = 2 * L
    src = [rng.integers(0, 256, (src_rows, S), dtype=np.uint8) for _ in range(P)]
    dst = [rng.integers(0, 256, (dst_rows, S), dtype=np.uint8) for _ in range(P)]
    src_idx = rng.integers(0, src_rows, n).astype(np.int64)
    dst_idx = rng.choice(dst_rows, size=n, replace=False).astype(np.int64)
    if n > 2:
        dst_idx[n - 1] = dst_rows  # a bad pair
    g_src = [torch.from_numpy(x).to(dev) for x in src]
    g_dst = [torch.from_numpy(x.copy()).to(dev) for x in dst]
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    _hs().transfer_kv_layers(g_src, g_dst, torch.from_numpy(src_idx).to(dev),
                             torch.from_numpy(dst_idx).to(dev), has_v=True, status=st)
    r_st = np.zeros(1, np.int32)
    oracle.transfer_kv(src_layers=src, dst_layers=dst, src_idx=src_idx, dst_idx=dst_idx,
                       status=r_st)
    torch.cuda.synchronize()
    for l in range(P):
        np.testing.assert_array_equal(g_dst[l].cpu().numpy(), dst[l], err_msg=f"layer {l}")
    assert st.item() == r_st[0]
