"""GPU parity for hs_fp8_store_kv against the CPU oracle, code by code: fp32,
fp16 and bf16 inputs; flat and paged caches; with and without scales; the
16-byte-chunk path and the element path (a head_dim that does not fill 16-byte
chunks); K only; out-of-range slots; special values (signed zeros,
subnormals, exact ties, finite overflow, infinities, NaN); and the full-size
write the benchmark times (4096 tokens of [8 x 128] bf16 K and V into 2^20-slot
caches, pages of 16), compared on sampled tokens."""
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


TORCH_DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def _as_oracle(t: torch.Tensor) -> np.ndarray:
    """Host copy in the oracle's input form (bf16 as its uint16 bits)."""
    t = t.cpu()
    return t.view(torch.uint16).numpy() if t.dtype == torch.bfloat16 else t.numpy()


def _specials(n, rng):
    base = np.array([0.0, -0.0, 1e-30, -1e-30, 2.0 ** -10, 3 * 2.0 ** -10, 2.0 ** -9,
                     1.0625, 1.1875, -1.0625, 447.9, 448.0, 463.0, 464.0, 465.0, 1e5, -1e5,
                     np.inf, -np.inf, np.nan, 0.0078125, 240.0, 232.0], np.float32)
    return np.resize(base, n) * np.where(rng.random(n) < 0.5, 1, 1).astype(np.float32)


def _run(dev, dtype, paged, scaled, T, Hh, D, ps, pages, with_v=True, specials=False, seed=0,
         head_step=1):
    hs = _hs()
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((T, 2 * Hh * head_step + 1, D)) * 40).astype(np.float32)
    if specials:
        flat = x.reshape(-1)
        idx = rng.choice(flat.size, size=flat.size // 3, replace=False)
        flat[idx] = _specials(idx.size, rng)
    xt = torch.from_numpy(x).to(TORCH_DT[dtype]).to(dev)
    # views of one buffer; head_step 2 spaces the heads out (head stride != dim)
    k = xt[:, : Hh * head_step : head_step]
    v = xt[:, Hh * head_step + 1:: head_step][:, :Hh]
    shape = (pages, ps, Hh, D) if paged else (pages * ps, Hh, D)
    kc = rng.integers(0, 256, shape, dtype=np.uint8)
    vc = rng.integers(0, 256, shape, dtype=np.uint8)
    loc = rng.choice(pages * ps, size=T, replace=False).astype(np.int64)
    loc[[1, T // 2]] = [pages * ps, -5]
    ks = vs = None
    if scaled:
        ks, vs = np.float32(0.37), np.float32(3.1)
    st_ref = np.zeros(1, np.int32)
    kc_ref, vc_ref = kc.copy(), vc.copy()
    oracle.fp8_store_kv(k=_as_oracle(k), v=_as_oracle(v) if with_v else None, k_cache=kc_ref,
                        v_cache=vc_ref if with_v else None, loc=loc, page_size=ps,
                        k_scale=ks, v_scale=vs, bf16=dtype == "bf16", status=st_ref)
    g_kc, g_vc = torch.from_numpy(kc).to(dev), torch.from_numpy(vc).to(dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    sc = (lambda a: None if a is None else torch.tensor([a], dtype=torch.float32, device=dev))
    hs.fp8_store_kv(k, v if with_v else None, g_kc, g_vc if with_v else None,
                    torch.from_numpy(loc).to(dev), k_scale=sc(ks), v_scale=sc(vs),
                    page_size=ps, status=st)
    torch.cuda.synchronize()
    for got, ref in ((g_kc.cpu().numpy(), kc_ref), (g_vc.cpu().numpy(), vc_ref)):
        nan_ref = (ref & 0x7F) == 0x7F
        nan_got = (got & 0x7F) == 0x7F
        np.testing.assert_array_equal(nan_got, nan_ref)
        np.testing.assert_array_equal(got[~nan_ref], ref[~nan_ref])
    assert st.item() == st_ref[0] == oracle.ST_BAD_INDEX


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("paged,scaled", [(True, True), (False, False), (True, False)])
def test_fp8_store_parity(dev, dtype, paged, scaled):
    _run(dev, dtype, paged, scaled, T=300, Hh=8, D=128, ps=16, pages=40, seed=hash(dtype) % 97)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_fp8_store_chunk_path_spaced_heads(dev, dtype):
    """Heads not contiguous in the input: the per-chunk kernel instead of the row kernel."""
    _run(dev, dtype, True, True, T=120, Hh=4, D=64, ps=8, pages=30, seed=21, head_step=2)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fp8_store_element_path(dev, dtype):
    _run(dev, dtype, True, True, T=77, Hh=3, D=13, ps=4, pages=30, seed=5)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_fp8_store_special_values(dev, dtype):
    _run(dev, dtype, True, True, T=64, Hh=2, D=64, ps=8, pages=16, specials=True, seed=9)
    _run(dev, dtype, False, False, T=64, Hh=2, D=64, ps=8, pages=16, specials=True, seed=10)


def test_fp8_store_k_only(dev):
    _run(dev, "bf16", True, False, T=50, Hh=4, D=32, ps=16, pages=8, with_v=False, seed=3)


def test_fp8_store_full_size_sampled(dev):
    """The benchmark's write: 4096 tokens x [8 x 128] bf16 K and V, 2^20-slot
    caches in pages of 16, scales given; 64 sampled tokens compared."""
    hs = _hs()
    T, Hh, D, ps, slots = 4096, 8, 128, 16, 1 << 20
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    k = torch.randn((T, Hh, D), generator=g, device=dev).to(torch.bfloat16)
    v = torch.randn((T, Hh, D), generator=g, device=dev).to(torch.bfloat16)
    kc = torch.zeros((slots // ps, ps, Hh, D), dtype=torch.uint8, device=dev)
    vc = torch.zeros_like(kc)
    loc = torch.randperm(slots, generator=g, device=dev)[:T]
    ks = torch.tensor([0.25], device=dev)
    vs = torch.tensor([1.5], device=dev)
    hs.fp8_store_kv(k, v, kc, vc, loc, k_scale=ks, v_scale=vs, page_size=ps)
    torch.cuda.synchronize()
    rng = np.random.default_rng(1)
    sample = rng.choice(T, size=64, replace=False)
    loc_h = loc.cpu().numpy()
    for kv, src, cache, sc in ((0, k, kc, 0.25), (1, v, vc, 1.5)):
        x = _as_oracle(src[torch.from_numpy(sample).to(dev)])
        ref = np.zeros((64, 1, Hh, D), np.uint8)
        oracle.fp8_store_kv(k=x, v=None, k_cache=ref, v_cache=None,
                            loc=np.arange(64, dtype=np.int64), page_size=1,
                            k_scale=np.float32(sc), bf16=True)
        got = cache.view(-1, Hh, D)[torch.from_numpy(loc_h[sample]).to(dev)].cpu().numpy()
        np.testing.assert_array_equal(got, ref[:, 0])
