"""Pins for the oracle's FP8 KV write (tokenspeed
tokenspeed_kernel/ops/kvcache/triton.py, fused_fp8_set_kv_buffer: K/V times
an inverse scale in fp32, converted to float8 e4m3 "fn", scattered to
cache_loc slots of a paged cache).

What fixes the encoder other than itself:
- every one of the 256 codes, decoded here from the format's definition
  (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, subnormals at
  exponent 0, S.1111.111 = NaN), encodes back to itself;
- the midpoint between every two neighbouring codes encodes to the code with
  the even mantissa, and values just either side of it to the nearer code;
- torch's float8_e4m3fn conversion (a library routine) agrees bit for bit on
  random values inside the finite range, subnormals included;
- finite overflow and infinities saturate to +-448 (the reading taken for the
  kernel's fp32 -> fp8 conversion), NaN stays NaN with its sign.
What fixes the store: numpy advanced-index assignment of torch-converted codes,
for fp32, fp16 and bf16 inputs, flat and paged layouts, with and without
scales; out-of-range slots are skipped with the status bit.  Planted mistakes
(ties away from zero; page and offset swapped) are caught.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle


def decode_e4m3(code: int) -> float:
    s = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 3) & 15, code & 7
    if e == 15 and m == 7:
        return math.copysign(float("nan"), s)
    if e == 0:
        return s * m * 2.0 ** -9
    return s * (1 + m / 8) * 2.0 ** (e - 7)


CODES = np.arange(256)
VALUES = np.array([decode_e4m3(int(c)) for c in CODES], dtype=np.float64)


def test_every_code_round_trips():
    enc = oracle.e4m3_encode(VALUES.astype(np.float32))
    nan = np.isnan(VALUES)
    np.testing.assert_array_equal(enc[~nan], CODES[~nan])
    assert set(enc[nan].tolist()) == {0x7F, 0xFF}
    assert oracle.e4m3_encode(np.array([0.0, -0.0], np.float32)).tolist() == [0x00, 0x80]


def _positive_ladder():
    # finite non-negative codes in increasing value order
    codes = [c for c in range(0x80) if not np.isnan(VALUES[c])]
    return sorted(codes, key=lambda c: VALUES[c])


def test_midpoints_round_to_even():
    lad = _positive_ladder()
    xs, want_mid = [], []
    for a, b in zip(lad, lad[1:]):
        mid = (VALUES[a] + VALUES[b]) / 2  # exact in fp32 for every e4m3 pair
        assert float(np.float32(mid)) == mid
        even = a if (a & 1) == 0 else b
        for sign in (1.0, -1.0):
            xs += [sign * mid, sign * np.nextafter(np.float32(mid), np.float32(0)),
                   sign * np.nextafter(np.float32(mid), np.float32(np.inf))]
            sb = 0x80 if sign < 0 else 0
            want_mid += [even | sb, a | sb, b | sb]
    got = oracle.e4m3_encode(np.array(xs, np.float32))
    np.testing.assert_array_equal(got, np.array(want_mid, np.uint8))


def test_matches_torch_in_range():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.uniform(-448, 448, 200_000),
        rng.standard_normal(200_000),
        rng.uniform(-2.0 ** -6, 2.0 ** -6, 100_000),           # subnormals
        np.ldexp(rng.uniform(1, 2, 50_000), rng.integers(-12, 9, 50_000)),
    ]).astype(np.float32)
    x = x[np.abs(x) < 464]  # torch turns larger magnitudes into NaN instead of saturating
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.e4m3_encode(x), ref)


def test_saturation_and_nan():
    big = np.array([448.0, 449.0, 463.9, 464.0, 465.0, 1e6, 3e38, np.inf], np.float32)
    got = oracle.e4m3_encode(np.concatenate([big, -big]))
    assert got.tolist() == [0x7E] * len(big) + [0xFE] * len(big)
    nan = np.array([np.nan, -np.nan], np.float32)
    nan[1] = -np.abs(nan[1])
    assert oracle.e4m3_encode(nan).tolist() == [0x7F, 0xFF]


def _expected_store(x_f32, inv, cache, loc, page_size, paged):
    y = torch.from_numpy(x_f32)
    if inv is not None:
        y = y * torch.tensor(inv, dtype=torch.float32)
    codes = y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    out = cache.copy()
    ok = (loc >= 0) & (loc < (out.shape[0] * (out.shape[1] if paged else 1)))
    if paged:
        out[loc[ok] // page_size, loc[ok] % page_size] = codes[ok]
    else:
        out[loc[ok]] = codes[ok]
    return out


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("paged,scaled", [(False, False), (True, True), (True, False)])
def test_store_matches_index_assignment(dtype, paged, scaled):
    rng = np.random.default_rng(hash((dtype, paged, scaled)) % 2**32)
    T, Hh, D, ps, pages = 37, 3, 20, 4, 30
    base = (rng.standard_normal((T, 2 * Hh + 1, D)) * 30).astype(np.float32)
    kf, vf = base[:, :Hh], base[:, Hh + 1:]          # strided head views
    if dtype == "f16":
        k_in, v_in = kf.astype(np.float16), vf.astype(np.float16)
        kx, vx = k_in.astype(np.float32), v_in.astype(np.float32)
    elif dtype == "bf16":
        kt = torch.from_numpy(np.ascontiguousarray(kf)).to(torch.bfloat16)
        vt = torch.from_numpy(np.ascontiguousarray(vf)).to(torch.bfloat16)
        k_in, v_in = kt.view(torch.uint16).numpy(), vt.view(torch.uint16).numpy()
        kx, vx = kt.float().numpy(), vt.float().numpy()
    else:
        k_in, v_in, kx, vx = kf, vf, kf, vf
    shape = (pages, ps, Hh, D) if paged else (pages * ps, Hh, D)
    kc = rng.integers(0, 256, shape, dtype=np.uint8)
    vc = rng.integers(0, 256, shape, dtype=np.uint8)
    loc = rng.choice(pages * ps, size=T, replace=False).astype(np.int64)
    loc[[4, 9]] = [pages * ps, -1]
    ks, vs = (np.float32(0.7), np.float32(2.5)) if scaled else (None, None)
    inv = (lambda sc: None if sc is None else np.float32(1) / sc)  # fp32 division
    ek = _expected_store(kx, inv(ks), kc, loc, ps, paged)
    ev = _expected_store(vx, inv(vs), vc, loc, ps, paged)
    st = np.zeros(1, np.int32)
    oracle.fp8_store_kv(k=k_in, v=v_in, k_cache=kc, v_cache=vc, loc=loc, page_size=ps,
                        k_scale=ks, v_scale=vs, bf16=dtype == "bf16", status=st)
    np.testing.assert_array_equal(kc, ek)
    np.testing.assert_array_equal(vc, ev)
    assert st[0] == oracle.ST_BAD_INDEX


def test_planted_fp8_mistakes_are_caught():
    lad = _positive_ladder()
    mids = np.array([(VALUES[a] + VALUES[b]) / 2 for a, b in zip(lad, lad[1:])], np.float32)
    evens = np.array([a if (a & 1) == 0 else b for a, b in zip(lad, lad[1:])], np.uint8)
    assert not np.array_equal(oracle.e4m3_encode(mids, mutant=13), evens)
    rng = np.random.default_rng(2)
    T, Hh, D, ps = 8, 2, 16, 4
    k = rng.standard_normal((T, Hh, D)).astype(np.float32)
    kc = np.zeros((10, ps, Hh, D), np.uint8)
    kc2 = kc.copy()
    loc = np.array([1, 5, 9, 14, 22, 30, 33, 38], np.int64)
    oracle.fp8_store_kv(k=k, v=None, k_cache=kc, v_cache=None, loc=loc, page_size=ps)
    oracle.fp8_store_kv(k=k, v=None, k_cache=kc2, v_cache=None, loc=loc, page_size=ps,
                        mutant=14)
    assert not np.array_equal(kc, kc2)
