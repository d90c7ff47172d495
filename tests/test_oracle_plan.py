"""Pins for the oracle's miss plan and its replay onto layers that share a
resolving layer's indices (vLLM csrc/libtorch_stable/hisparse_kernels.cu,
hisparse_gather_plan_kernel and hisparse_gather_compact_kernel: shared layers
see the same indices and slot assignment, so only their bytes differ).

- the plan (miss pool rows, hot rows, entry mask) equals the brute force's,
  exhaustively on tiny inputs and on random cases with host-injected corruption;
- replaying layer A's plan onto layer B (same state, other bytes) gives exactly
  the hot buffer a full resolution of layer B gives;
- consistency with the call's own outputs: mask count = miss count, plan
  entries follow the masked entries in top-k order, dst = out, src =
  pool_rows[r][id], entries past the miss count untouched;
- the replay's bounds: no-row misses, bad indices, clamped counts;
- planted mistakes in the plan and in the replay are caught.
"""
from __future__ import annotations

import itertools

import numpy as np
import pytest

import cases
import oracle


def _plan_prefix(src, dst, miss):
    return [(list(map(int, src[b, : miss[b]])), list(map(int, dst[b, : miss[b]])))
            for b in range(src.shape[0])]


def _compare_plan(case: cases.Case, what, mutant=0):
    a, b = case.copy(), case.copy()
    out, miss, _, _, src, dst, mask = cases.run_oracle(a, mutant=mutant, plan=True)
    plans = []
    cases.run_brute(b, plans=plans)
    for r, pl in enumerate(plans):
        assert list(map(int, src[r, : miss[r]])) == pl["src"], f"src row {r} {what}"
        assert list(map(int, dst[r, : miss[r]])) == pl["dst"], f"dst row {r} {what}"
        assert list(map(int, mask[r])) == pl["mask"], f"mask row {r} {what}"
    return a


def plan_exhaustive(mutant=0):
    rng = np.random.default_rng(21)
    for H in range(1, 5):
        for K in range(1, min(H, 3) + 1):
            base = cases.random_case(rng, B=1, K=K, H=H, S=3, R=1, seq_len=6, P=8, cols=6)
            for _ in range(2):
                base.topk = rng.integers(-1, 6, size=(1, K)).astype(np.int32)
                cases.run_oracle(base)
            for ids in itertools.product(range(-1, 7), repeat=K):
                c = base.copy()
                c.topk = np.array([ids], dtype=np.int32)
                _compare_plan(c, f"H={H} ids={ids}", mutant)


def plan_random(mutant=0, seeds=range(60)):
    for seed in seeds:
        rng = np.random.default_rng(5000 + seed)
        H = int(rng.integers(1, 13))
        K = int(rng.integers(1, H + 1))
        B = int(rng.integers(1, 5))
        seq = rng.integers(1, 4 * H + 3, size=B)
        c = cases.random_case(rng, B=B, K=K, H=H, S=int(rng.choice([1, 4, 16])), R=B + 2,
                              seq_len=seq, P=int(rng.integers(4 * H + 3, 8 * H + 8)))
        c.num_real = int(rng.choice([-1, B, max(0, B - 1)]))
        prev = None
        for step in range(5):
            c.topk = prev = cases.random_ids(rng, c, prev=prev)
            if step >= 2:
                cases.corrupt(np.random.default_rng(seed * 17 + step), c)
            c = _compare_plan(c, f"seed={seed} step={step}", mutant)


def test_plan_matches_brute_exhaustive():
    plan_exhaustive()


def test_plan_matches_brute_random_with_corruption():
    plan_random()


def replay_equals_resolution(mutant=0, with_v=False, seeds=range(12), corrupt=True):
    """Layers A and B share state; B's bytes differ.  Resolving B must equal
    replaying A's plan onto B's pool and B's previous hot buffer."""
    for seed in seeds:
        rng = np.random.default_rng(900 + seed)
        H = int(rng.integers(4, 40))
        K = int(rng.integers(1, H + 1))
        B = int(rng.integers(1, 5))
        A = cases.random_case(rng, B=B, K=K, H=H, S=int(rng.choice([3, 16, 20])), R=B + 1,
                              seq_len=rng.integers(H // 2, 6 * H, size=B), with_v=with_v)
        Bl = A.copy()
        Bl.pool_k = rng.integers(0, 256, size=A.pool_k.shape, dtype=np.uint8)
        Bl.hot_k = rng.integers(0, 256, size=A.hot_k.shape, dtype=np.uint8)
        if with_v:
            Bl.pool_v = rng.integers(0, 256, size=A.pool_v.shape, dtype=np.uint8)
            Bl.hot_v = rng.integers(0, 256, size=A.hot_v.shape, dtype=np.uint8)
        prev = None
        for step in range(6):
            ids = cases.random_ids(rng, A, prev=prev)
            prev = ids
            if corrupt and step >= 3:
                cases.corrupt(np.random.default_rng(seed * 7 + step), A)
                Bl.tokens[:], Bl.lru[:], Bl.pool_rows[:] = A.tokens, A.lru, A.pool_rows
                Bl.rows[:], Bl.req_state[:] = A.rows, A.req_state
            A.topk, Bl.topk = ids, ids.copy()
            out, miss, _, _, src, dst, _ = cases.run_oracle(A, mutant=mutant, plan=True)
            hot_k, hot_v = Bl.hot_k.copy(), (Bl.hot_v.copy() if with_v else None)
            st = np.zeros(1, np.int32)
            oracle.gather_misses(pool_k=Bl.pool_k, pool_v=Bl.pool_v, hot_k=hot_k, hot_v=hot_v,
                                 miss_src=src, miss_dst=dst, miss_count=miss, status=st,
                                 mutant=mutant)
            out_b, miss_b, _, _ = cases.run_oracle(Bl)
            np.testing.assert_array_equal(out, out_b)
            np.testing.assert_array_equal(miss, miss_b)
            np.testing.assert_array_equal(hot_k, Bl.hot_k, err_msg=f"seed={seed} step={step}")
            if with_v:
                np.testing.assert_array_equal(hot_v, Bl.hot_v)
            assert st[0] == 0


@pytest.mark.parametrize("with_v", [False, True])
def test_replay_equals_resolution(with_v):
    replay_equals_resolution(with_v=with_v)


def test_plan_consistent_with_outputs():
    rng = np.random.default_rng(3)
    c = cases.random_case(rng, B=4, K=50, H=120, S=8, R=5, seq_len=900)
    prev = None
    for step in range(6):
        c.topk = prev = cases.random_ids(rng, c, prev=prev)
        ids, req = c.topk.copy(), c.req_state.copy()
        pool_rows = c.pool_rows.copy()
        out, miss, _, _, src, dst, mask = cases.run_oracle(c, plan=True)
        for b in range(c.B):
            masked = np.flatnonzero(mask[b])
            assert set(np.unique(mask[b])) <= {0, 1}
            assert len(masked) == miss[b]
            np.testing.assert_array_equal(dst[b, : miss[b]], out[b, masked])
            np.testing.assert_array_equal(src[b, : miss[b]], pool_rows[req[b], ids[b, masked]])
            assert np.all(src[b, miss[b]:] == cases.PLAN_FILL_SRC)
            assert np.all(dst[b, miss[b]:] == cases.PLAN_FILL_DST)


def test_gather_bounds():
    S = 4
    pool = np.arange(10 * S, dtype=np.uint8).reshape(10, S)
    hot = np.zeros((6, S), np.uint8)
    src = np.array([[2, 11, 4, 5, 7], [1, 1, 1, 1, 1], [3, 9, 0, 0, 0]], np.int64)
    dst = np.array([[0, 1, -1, 6, 2], [5, 5, 5, 5, 5], [3, 4, 0, 0, 0]], np.int32)
    count = np.array([5, -2, 9], np.int32)  # row 1: none; row 2: clamped to top_k = 5
    st = np.zeros(1, np.int32)
    oracle.gather_misses(pool_k=pool, hot_k=hot, miss_src=src, miss_dst=dst, miss_count=count,
                         status=st)
    exp = np.zeros((6, S), np.uint8)
    exp[0], exp[2] = pool[2], pool[7]          # row 0: pair 1 bad src, 2 no row, 3 bad dst
    exp[3], exp[4] = pool[3], pool[9]          # row 2: all five (dst 0 gets pool 0 last)
    exp[0] = pool[0]
    np.testing.assert_array_equal(hot, exp)
    assert st[0] == oracle.ST_BAD_INDEX


@pytest.mark.parametrize("mutant,check", [
    (11, lambda: replay_equals_resolution(11, seeds=range(4), corrupt=False)),
    (12, lambda: plan_random(12, seeds=range(10))),
])
def test_planted_plan_mistakes_are_caught(mutant, check):
    with pytest.raises(AssertionError):
        check()
