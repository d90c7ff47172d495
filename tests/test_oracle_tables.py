"""Pins for the oracle's block-table translation, resident-block lookup and
invalidation of rewritten tokens (vLLM csrc/libtorch_stable/hisparse_kernels.cu:
hisparse_resolve_residency_kernel, Phase 1; hisparse_invalidate_written_slots_kernel).

- translation: pools are laid out block by block through numpy reshapes, each row
  holding the bytes of (state row, token); after every step every emitted hot row
  holds the bytes of the token it was asked for;
- a token whose source block is unmapped behaves exactly like an invalid id;
- a token of a resident block is served from the resident cache and otherwise
  behaves exactly like an invalid id (not looked up, not counted);
- the source table gives the same results as the equivalent pool_rows table;
- invalidation equals numpy masked assignment on slots [0, H), slot H untouched;
- planted mistakes (block 0 taken as mapped; slot H invalidated) are caught.
"""
from __future__ import annotations

import numpy as np
import pytest

import cases
import oracle

S = 16


def _row_bytes(r, t):
    b = np.zeros(S, np.uint8)
    b[:4] = np.frombuffer(np.int32(r).tobytes(), np.uint8)
    b[4:8] = np.frombuffer(np.int32(t).tobytes(), np.uint8)
    b[8:] = (r * 7 + t * 13) % 251
    return b


def block_case(rng, *, B=3, K=24, H=40, L=200, bs=4, unmapped=0.0):
    """A case whose pool is addressed through a source block table."""
    R = B + 1
    nb = -(-L // bs)
    phys = rng.permutation(R * nb) + 1            # block 0 is the null block
    src = phys.reshape(R, nb).astype(np.int32)
    if unmapped:
        src[rng.random(src.shape) < unmapped] = 0
    pool = np.zeros((R * nb + 1, bs, S), np.uint8)   # block-major view of the pool
    for r in range(R):
        for j in range(nb):
            for k in range(bs):
                pool[phys[r * nb + j], k] = _row_bytes(r, j * bs + k)
    c = cases.random_case(rng, B=B, K=K, H=H, S=S, R=R, seq_len=L, P=8, cols=L)
    c.pool_k = pool.reshape(-1, S)
    c.pool_rows = np.full((R, L), -7, np.int64)       # unused with a source table
    c.tables = dict(src_block_table=src, src_block_size=bs)
    return c


def _check_bytes(c, out, ids):
    for b in range(c.B):
        r = int(c.req_state[b])
        for i, t in enumerate(ids[b]):
            if out[b, i] >= 0 and 0 <= t < c.seq_lens[b] - 1:
                np.testing.assert_array_equal(c.hot_k[out[b, i]], _row_bytes(r, int(t)))


def test_translation_fetches_the_right_rows():
    rng = np.random.default_rng(1)
    c = block_case(rng)
    prev = None
    for step in range(6):
        ids = cases.random_ids(rng, c, prev=prev, p_invalid=0.05, p_dup=0.05)
        prev = ids
        c.topk = ids
        out, miss, status, _ = cases.run_oracle(c)
        assert miss.sum() > 0 or step > 0
        _check_bytes(c, out, ids)


def _strip(ids, mask):
    x = ids.copy()
    x[mask] = -1
    return x


@pytest.mark.parametrize("mutant", [0, 15])
def test_unmapped_blocks_behave_like_invalid_ids(mutant):
    rng = np.random.default_rng(2)
    a = block_case(rng, unmapped=0.2)
    src, bs = a.tables["src_block_table"], a.tables["src_block_size"]
    b = a.copy()
    prev = None
    for step in range(5):
        ids = cases.random_ids(rng, a, prev=prev, p_invalid=0.0, p_dup=0.0)
        prev = ids
        rows = a.req_state[:, None]
        blk = np.clip(ids // bs, 0, src.shape[1] - 1)
        # the newest token lives in slot H and needs no source row
        unm = (ids >= 0) & (src[rows, blk] <= 0) & (ids != a.seq_lens[:, None] - 1)
        a.topk, b.topk = ids, _strip(ids, unm)
        ra = cases.run_oracle(a, mutant=mutant)
        rb = cases.run_oracle(b)
        if mutant:
            if not all(np.array_equal(x, y) for x, y in zip(ra, rb)):
                return
            continue
        for x, y in zip(ra, rb):
            np.testing.assert_array_equal(x, y)
        cases.assert_same_state(a, b, f"step {step}")
    if mutant:
        pytest.fail("the planted mistake was not caught")


def test_source_table_equals_pool_rows():
    rng = np.random.default_rng(3)
    a = block_case(rng)
    src, bs = a.tables["src_block_table"], a.tables["src_block_size"]
    b = a.copy()
    R, L = a.pool_rows.shape
    # the same map written as a per-token table: block-major pool rows
    pool_idx = np.arange(a.pool_k.shape[0]).reshape(-1, bs)
    b.pool_rows = np.stack([pool_idx[src[r, np.arange(L) // bs], np.arange(L) % bs]
                            for r in range(R)]).astype(np.int64)
    b.tables = {}
    prev = None
    for step in range(5):
        ids = cases.random_ids(rng, a, prev=prev)
        prev = ids
        a.topk, b.topk = ids, ids.copy()
        for x, y in zip(cases.run_oracle(a, plan=True), cases.run_oracle(b, plan=True)):
            np.testing.assert_array_equal(x, y)
        cases.assert_same_state(a, b, f"step {step}")


def test_resident_blocks_are_served_directly():
    rng = np.random.default_rng(4)
    a = block_case(rng)
    R, L = a.pool_rows.shape
    rbs, nb = 8, -(-L // 8)
    res = np.full((R, nb), -1, np.int32)
    null = 5
    pick = rng.random((R, nb)) < 0.3
    res[pick] = rng.permutation(1000)[: pick.sum()] + 10
    res[0, 0] = null                                   # the null block is not resident
    a.tables.update(res_block_table=res, res_block_size=rbs, res_null_block=null)
    b = a.copy()
    b.tables = {k: v for k, v in a.tables.items() if not k.startswith("res")}
    dev_rows = np.arange(2000 * rbs).reshape(2000, rbs)   # resident cache rows, block-major
    prev = None
    for step in range(5):
        ids = cases.random_ids(rng, a, prev=prev, p_dup=0.0)
        prev = ids
        rows = a.req_state[:, None]
        e = res[rows, np.clip(ids // rbs, 0, nb - 1)]
        valid = (ids >= 0) & (ids < a.seq_lens[:, None])
        resident = valid & (e >= 0) & (e != null)
        a.topk, b.topk = ids, _strip(ids, resident)
        out_a, miss_a, st_a, stats_a = cases.run_oracle(a)
        out_b, miss_b, st_b, stats_b = cases.run_oracle(b)
        first = np.zeros_like(resident)  # a repeated resident id: only its first copy is served
        for r in range(ids.shape[0]):
            seen = set()
            for i, t in enumerate(ids[r]):
                first[r, i] = valid[r, i] and t not in seen
                if valid[r, i]:
                    seen.add(int(t))
        served = resident & first
        want = out_b.copy()
        want[served] = dev_rows[e[served], ids[served] % rbs]
        np.testing.assert_array_equal(out_a, want)
        np.testing.assert_array_equal(miss_a, miss_b)
        np.testing.assert_array_equal(stats_a, stats_b)
        cases.assert_same_state(a, b, f"step {step}")


def test_resident_before_newest_and_fast_path():
    rng = np.random.default_rng(5)
    c = block_case(rng, B=2, K=6, H=40, L=200)
    c.seq_lens[1] = 30                                   # row 1 takes the fast path
    R = c.pool_rows.shape[0]
    res = np.full((R, 25), -1, np.int32)
    r0, r1 = int(c.req_state[0]), int(c.req_state[1])
    res[r0, 199 // 8] = 3                                # the newest token's block
    res[r1, 1] = 4                                       # tokens 8..15 of row 1
    c.tables.update(res_block_table=res, res_block_size=8, res_null_block=-1)
    c.topk = np.array([[199, 5, 7, -1, 3, 199], [9, 20, 40, 15, 2, 9]], np.int32)
    out, *_ = cases.run_oracle(c)
    assert out[0, 0] == 3 * 8 + 199 % 8 and out[0, 5] == -1     # resident; later copy dup
    assert out[1, 0] == 4 * 8 + 1 and out[1, 3] == 4 * 8 + 7     # fast path, resident
    assert out[1, 1] == c.rows[r1, 20] and out[1, 2] == -1        # fast path, ordinary
    assert out[1, 5] == 4 * 8 + 1                                  # fast path keeps repeats


@pytest.mark.parametrize("mutant", [0, 16])
def test_invalidation_matches_masked_assignment(mutant):
    rng = np.random.default_rng(6)
    R, H = 5, 30
    tok = rng.integers(-1, 40, (R, H + 3)).astype(np.int32)
    rows = np.array([0, 2, 2, -1, 4, 7, 1], np.int64)
    toks = np.array([5, 11, 3, 5, -2, 6, 77], np.int32)
    tok[1, H] = 77  # only slot H of row 1 holds token 77: it must stay
    exp = tok.copy()
    for r, t in zip(rows, toks):
        if r < 0 or t < 0 or r >= R:
            continue
        part = exp[r, :H]
        part[part == t] = -1
    st = np.zeros(1, np.int32)
    got = tok.copy()
    if mutant:
        lib = oracle.load(mutant)
        import ctypes as C
        lib.hso_invalidate_tokens(got.ctypes.data, got.strides[0] // 4, H, R, rows.ctypes.data,
                                  toks.ctypes.data, len(toks), st.ctypes.data)
        assert not np.array_equal(got, exp)
        return
    oracle.invalidate_tokens(slot_tokens=got, hot_size=H, state_rows=rows, tokens=toks,
                             status=st)
    np.testing.assert_array_equal(got, exp)
    assert st[0] == oracle.ST_BAD_INDEX
