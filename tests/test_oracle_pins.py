"""Pins for the CPU oracle's swap-in: what fixes it other than itself.

- a hand-worked example and hand-worked tripwire cases (tests/golden/);
- brute force on tiny inputs, exhaustive over small id tuples and random with
  host-injected corruption (tests/brute.py: list scans, no hashing, and the
  LRU writeback computed with both pages' index formulas);
- closed forms: full reuse is a fixed point; all-fresh ids from a cold start
  land in slot (s*K + i) mod H; M = K - hits - newest - invalid - dup - badpool;
- a textbook LRU cache (functools.lru_cache) at top_k = 1;
- invariants on larger seeded workloads;
- planted mistakes (oracle built with HSO_MUTANT=k) are caught by these pins.
"""
from __future__ import annotations

import functools
import itertools
import json
import os

import numpy as np
import pytest

import cases
import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ------------------------------------------------------------------ golden
def _golden_case(H, seq_len, rows, tokens, lru, pool_rows, P, hot_num_rows, S=2):
    R = 1
    W = H + 1
    tok = np.full((R, W), -1, dtype=np.int32)
    tok[0, : len(tokens)] = tokens
    rr = np.full((R, W), -1, dtype=np.int32)
    rr[0, : len(rows)] = rows
    lr = np.array([lru], dtype=np.int16)
    # a few spare rows past P keep a planted off-by-one read inside the buffer
    pool_k = np.array([[x % 256, (x + 1) % 256] for x in range(P + 4)], dtype=np.uint8)[:P]
    hot_k = np.full((hot_num_rows, S), 0xEE, dtype=np.uint8)
    return cases.Case(H=H, K=0, S=S, topk=np.zeros((1, 0), np.int32),
                      seq_lens=np.array([seq_len], np.int64), req_state=np.zeros(1, np.int64),
                      tokens=tok, rows=rr, lru=lr, pool_rows=np.array([pool_rows], np.int64),
                      pool_k=pool_k, pool_v=None, hot_k=hot_k, hot_v=None)


def _check_golden_steps(case, steps, mutant=0):
    for n, st in enumerate(steps):
        case.topk = np.array([st["ids"]], dtype=np.int32)
        case.K = case.topk.shape[1]
        out, miss, status, _ = cases.run_oracle(case, mutant=mutant)
        assert out[0].tolist() == st["out"], f"step {n} out"
        assert int(miss[0]) == st["miss_count"], f"step {n} miss_count"
        assert int(status[0]) == st["status"], f"step {n} status"
        assert case.lru[0].tolist() == st["lru"], f"step {n} lru"
        assert case.tokens[0, : len(st["tokens"])].tolist() == st["tokens"], f"step {n} tokens"
        for hr, pr in st["hot_rows_from_pool"].items():
            assert case.hot_k[int(hr)].tolist() == case.pool_k[pr].tolist(), f"step {n} row {hr}"


def golden_worked_example(mutant=0):
    g = json.load(open(os.path.join(GOLDEN, "swap_in_worked_example.json")))
    H, L = g["hot_size"], g["seq_len"]
    case = _golden_case(H, L, g["slot_rows"], [-1] * (H + 1), list(range(H)),
                        [50 + t for t in range(L)], 64, 105)
    _check_golden_steps(case, g["steps"], mutant)


def golden_tripwires(mutant=0):
    g = json.load(open(os.path.join(GOLDEN, "swap_in_tripwires.json")))
    c0, c1 = g["cases"]
    case = _golden_case(c0["hot_size"], c0["seq_len"], c0["rows"], c0["tokens"], c0["lru"],
                        list(range(c0["seq_len"])), c0["pool_num_rows"], c0["hot_num_rows"])
    _check_golden_steps(case, c0["steps"], mutant)
    pr = list(range(c1["seq_len"]))
    pr[4] = c1["pool_num_rows"]  # exactly one past the last pool row
    case = _golden_case(c1["hot_size"], c1["seq_len"], c1["rows"], c1["tokens"], c1["lru"],
                        pr, c1["pool_num_rows"], c1["hot_num_rows"])
    _check_golden_steps(case, c1["steps"], mutant)


def test_golden_worked_example():
    golden_worked_example()


def test_golden_tripwires():
    golden_tripwires()


# ------------------------------------------------------------------ brute force
def _compare_step(c_or: cases.Case, c_br: cases.Case, what, mutant=0):
    o1 = cases.run_oracle(c_or, mutant=mutant)
    o2 = cases.run_brute(c_br)
    for name, x, y in zip(("out", "miss_count", "status", "stats"), o1, o2):
        np.testing.assert_array_equal(x, y, err_msg=f"{name} {what}")
    cases.assert_same_state(c_or, c_br, what)


def brute_exhaustive(mutant=0, max_k=3):
    """Every id tuple over [-1, 7) for K <= max_k, from a warmed state, seq_len 6
    (ids 5 = newest, 6 = invalid)."""
    rng = np.random.default_rng(7)
    for H in range(1, 5):
        for K in range(1, min(H, max_k) + 1):
            base = cases.random_case(rng, B=1, K=K, H=H, S=3, R=1, seq_len=6, P=8, cols=6)
            # warm the state with two random steps
            for _ in range(2):
                base.topk = rng.integers(-1, 6, size=(1, K)).astype(np.int32)
                cases.run_oracle(base)
            for ids in itertools.product(range(-1, 7), repeat=K):
                a = base.copy()
                a.topk = np.array([ids], dtype=np.int32)
                _compare_step(a, a.copy(), f"H={H} ids={ids}", mutant)


def brute_random(mutant=0, seeds=range(150), corrupt=True):
    for seed in seeds:
        rng = np.random.default_rng(1000 + seed)
        H = int(rng.integers(1, 13))
        K = int(rng.integers(1, H + 1))
        B = int(rng.integers(1, 5))
        S = int(rng.choice([1, 3, 4, 16, 17]))
        seq = rng.integers(1, 4 * H + 3, size=B)
        a = cases.random_case(rng, B=B, K=K, H=H, S=S, R=B + 2, seq_len=seq,
                              P=int(rng.integers(4 * H + 3, 8 * H + 8)))
        a.num_real = int(rng.choice([-1, B, max(0, B - 1)]))
        b = a.copy()
        prev = None
        for step in range(5):
            ids = cases.random_ids(rng, a, prev=prev)
            prev = ids
            a.topk = ids
            b.topk = ids.copy()
            if corrupt and step >= 2:
                r2 = np.random.default_rng(seed * 31 + step)
                cases.corrupt(r2, a)
                cases.corrupt(np.random.default_rng(seed * 31 + step), b)
            _compare_step(a, b, f"seed={seed} step={step}", mutant)


def test_brute_exhaustive_tiny():
    brute_exhaustive()


def test_brute_random_with_corruption():
    brute_random()


# ------------------------------------------------------------------ closed forms
def _clean_case(rng, B, K, H, seq_len, S=8):
    return cases.random_case(rng, B=B, K=K, H=H, S=S, R=B, seq_len=seq_len)


def closed_form_fixed_point(mutant=0):
    """Full reuse: after the first step the state is a fixed point, M = 0 and
    no byte moves."""
    rng = np.random.default_rng(11)
    for H, K in ((8, 8), (16, 5), (64, 16), (33, 32)):
        c = _clean_case(rng, 3, K, H, seq_len=10 * H)
        ids = np.stack([rng.choice(10 * H - 1, size=K, replace=False) for _ in range(3)])
        c.topk = ids.astype(np.int32)
        cases.run_oracle(c, mutant)
        lru0, tok0, hot0 = c.lru.copy(), c.tokens.copy(), c.hot_k.copy()
        out0 = None
        for _ in range(3):
            c.topk = np.stack([rng.permutation(r) for r in ids]).astype(np.int32)
            out, miss, status, stats = cases.run_oracle(c, mutant)
            assert np.all(miss == 0) and np.all(status == 0)
            assert int(stats[0]) == 3 * K and int(stats[1]) == 0
            np.testing.assert_array_equal(c.lru, lru0)
            np.testing.assert_array_equal(c.tokens, tok0)
            np.testing.assert_array_equal(c.hot_k, hot0)
            # every entry resolves to the hot row that its token occupies
            srt = np.sort(out, axis=1)
            if out0 is not None:
                np.testing.assert_array_equal(srt, out0)
            out0 = srt


def closed_form_cold_fresh(mutant=0):
    """All-fresh, never-resident ids from a cold start with H % K == 0: the i-th
    entry of step s lands in slot (s*K + i) mod H."""
    rng = np.random.default_rng(12)
    for H, K in ((8, 2), (12, 4), (64, 16), (6, 6)):
        L = 50 * H
        c = _clean_case(rng, 2, K, H, seq_len=L)
        fresh = [rng.permutation(L - 1) for _ in range(2)]  # never the newest token
        for s in range(3 * H // K):
            c.topk = np.stack([f[s * K:(s + 1) * K] for f in fresh]).astype(np.int32)
            out, miss, status, _ = cases.run_oracle(c, mutant)
            assert np.all(miss == K) and np.all(status == 0)
            for b in range(2):
                r = int(c.req_state[b])
                want = [int(c.rows[r, (s * K + i) % H]) for i in range(K)]
                assert out[b].tolist() == want, (H, K, s, b)
                for i in range(K):
                    t = int(c.topk[b, i])
                    np.testing.assert_array_equal(c.hot_k[want[i]], c.pool_k[c.pool_rows[r, t]])


def closed_form_miss_identity(mutant=0):
    """M = K - hits - newest - invalid - dup - badpool on random rows."""
    rng = np.random.default_rng(13)
    for seed in range(40):
        H = int(rng.integers(4, 40))
        K = int(rng.integers(1, H + 1))
        c = _clean_case(rng, 3, K, H, seq_len=int(rng.integers(H + 1, 4 * H)))
        P = c.pool_k.shape[0]
        prev = None
        for step in range(4):
            ids = cases.random_ids(rng, c, prev=prev)
            prev = ids
            c.topk = ids
            if step == 3:
                c.pool_rows[:, rng.integers(c.pool_rows.shape[1], size=3)] = P + 1
            tok_before = c.tokens.copy()
            out, miss, status, stats = cases.run_oracle(c, mutant)
            total_hits = 0
            for b in range(3):
                L = int(c.seq_lens[b])
                r = int(c.req_state[b])
                row = [int(x) for x in ids[b]]
                invalid = sum(1 for t in row if not (0 <= t < L))
                firsts, dup = [], 0
                for t in row:
                    if 0 <= t < L:
                        if t in firsts:
                            dup += 1
                        else:
                            firsts.append(t)
                newest = sum(1 for t in firsts if t == L - 1)
                wanted = [t for t in firsts if t != L - 1]
                resident = set(int(x) for x in tok_before[r, :c.H])
                hits = sum(1 for t in wanted if t in resident)
                bad = sum(1 for t in wanted
                          if t not in resident and not (0 <= c.pool_rows[r, t] < P))
                total_hits += hits
                assert int(miss[b]) == K - hits - newest - invalid - dup - bad
            assert int(stats[0]) == total_hits


def lru_cache_k1(mutant=0):
    """top_k = 1: the swap-in is a plain LRU cache of capacity H; its hit/miss
    sequence equals functools.lru_cache(maxsize=H) on the same id stream."""
    rng = np.random.default_rng(14)
    for H in (1, 2, 3, 7, 16):
        L = 4 * H + 9
        c = _clean_case(rng, 1, 1, H, seq_len=L)
        stream = rng.integers(0, L - 1, size=300)  # never the newest token

        @functools.lru_cache(maxsize=H)
        def fetch(t):
            return t

        for t in stream:
            before = fetch.cache_info().misses
            fetch(int(t))
            textbook_miss = fetch.cache_info().misses - before
            c.topk = np.array([[t]], dtype=np.int32)
            _, miss, _, _ = cases.run_oracle(c, mutant)
            assert int(miss[0]) == textbook_miss, (H, t)


def test_closed_form_fixed_point():
    closed_form_fixed_point()


def test_closed_form_cold_fresh_slots():
    closed_form_cold_fresh()


def test_closed_form_miss_identity():
    closed_form_miss_identity()


def test_textbook_lru_cache_at_top_k_1():
    lru_cache_k1()


# ------------------------------------------------------------------ invariants
def check_invariants(c: cases.Case, prev_hot, out, miss):
    H = c.H
    for b in range(c.B):
        r = int(c.req_state[b])
        if r < 0 or r >= c.lru.shape[0]:
            continue
        L = int(c.seq_lens[b])
        lru = c.lru[r, :H].astype(np.int64)
        assert sorted(lru.tolist()) == list(range(H)), "lru is not a permutation"
        res = c.tokens[r, :H]
        res = res[res >= 0]
        assert len(np.unique(res)) == len(res), "duplicate resident token"
        if L > H:
            for t in set(int(x) for x in c.topk[b]):
                if 0 <= t < L - 1:
                    assert t in set(res.tolist()), "requested id not resident"
        o = out[b][out[b] >= 0]
        assert len(np.unique(o)) == len(o), "repeated hot row in one output row"
        for i in range(c.K):
            t = int(c.topk[b, i])
            if out[b, i] >= 0 and L > H and t != L - 1:
                np.testing.assert_array_equal(c.hot_k[out[b, i]], c.pool_k[c.pool_rows[r, t]])
    return prev_hot


def test_invariants_seeded_workload():
    rng = np.random.default_rng(15)
    for H, K, reuse in ((64, 16, 0.5), (256, 128, 0.9), (128, 128, 0.3)):
        L = 16 * H
        c = cases.random_case(rng, B=3, K=K, H=H, S=20, R=4, seq_len=L)
        ts = synth.TopkStream(99, 0, 3, K, L, reuse)
        for step in range(12):
            c.topk = ts.next()
            prev_hot = c.hot_k.copy()
            out, miss, status, _ = cases.run_oracle(c)
            assert np.all(status == 0)
            check_invariants(c, prev_hot, out, miss)
            # bytes outside the rows written by misses are unchanged
            written = set()
            for b in range(3):
                r = int(c.req_state[b])
                hit_or_new = set()
                for i in range(K):
                    if out[b, i] >= 0:
                        hit_or_new.add(int(out[b, i]))
                written |= hit_or_new
            untouched = np.array(sorted(set(range(c.hot_k.shape[0])) - written))
            np.testing.assert_array_equal(c.hot_k[untouched], prev_hot[untouched])


# ------------------------------------------------------------------ planted mistakes
MUTANTS = {
    1: "hits written before misses in the LRU order",
    2: "misses take most-recently-used evictables",
    3: "repeated id: last occurrence wins",
    4: "newest token not bound to the newest slot",
    5: "fast path only for seq_len < H",
    6: "copy reads pool row = token id instead of pool_rows[token]",
    7: "hits reversed in the LRU order",
    8: "pool row bound off by one",
    9: "miss_count excludes tripwired misses",
    10: "fast path ignores min(seq_len, top_k)",
}

PIN_BATTERY = [
    ("golden", golden_worked_example),
    ("tripwires", golden_tripwires),
    ("brute_exhaustive", lambda m: brute_exhaustive(m, max_k=2)),
    ("brute_random", lambda m: brute_random(m, seeds=range(60))),
    ("fixed_point", closed_form_fixed_point),
    ("cold_fresh", closed_form_cold_fresh),
    ("lru_cache", lru_cache_k1),
]


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_planted_mistake_is_caught(mutant):
    """Build the oracle with one planted mistake; at least one pin must fail."""
    caught = []
    for name, fn in PIN_BATTERY:
        try:
            fn(mutant)
        except AssertionError:
            caught.append(name)
    assert caught, f"mutant {mutant} ({MUTANTS[mutant]}) passed every pin"


def test_sequence_bound_makes_bad_state_rows():
    """A row longer than max_seq_len is rejected exactly like a state row past the
    table (R7): -1, no miss, HS_ST_BAD_STATE, state untouched; other rows as usual."""
    rng = np.random.default_rng(12)
    a = cases.random_case(rng, B=3, K=20, H=50, S=4, R=4, seq_len=400)
    a.seq_lens[1] = 600
    b = a.copy()
    a.max_seq_len = 500
    b.req_state[1] = 99                        # the reference: a state row past the table
    before = a.copy()
    for step in range(3):
        ids = cases.random_ids(rng, a)
        a.topk, b.topk = ids, ids.copy()
        ra, rb = cases.run_oracle(a), cases.run_oracle(b)
        for x, y in zip(ra, rb):
            np.testing.assert_array_equal(x, y)
        assert ra[2][1] == oracle.ST_BAD_STATE
    r1 = int(before.req_state[1])
    np.testing.assert_array_equal(a.tokens[r1], before.tokens[r1])
    np.testing.assert_array_equal(a.lru[r1], before.lru[r1])
