"""Seeded swap-in cases (numpy, host memory) shared by the oracle pins and the
GPU parity tests.  Holds no swap-in arithmetic: it builds inputs and state,
optionally corrupts state on the host, and compares results."""
from __future__ import annotations

import dataclasses

import numpy as np

import synth


@dataclasses.dataclass
class Case:
    H: int
    K: int
    S: int
    topk: np.ndarray        # int32 [B, K]
    seq_lens: np.ndarray    # int64 [B]
    req_state: np.ndarray   # int64 [B]
    tokens: np.ndarray      # int32 [R, W]
    rows: np.ndarray        # int32 [R, W]
    lru: np.ndarray         # int16 [R, H]
    pool_rows: np.ndarray   # int64 [R, cols]
    pool_k: np.ndarray      # uint8 [P, S]
    pool_v: np.ndarray | None
    hot_k: np.ndarray       # uint8 [hot_rows, S]
    hot_v: np.ndarray | None
    num_real: int = -1
    max_seq_len: int = 0  # 0, or a bound on seq_lens (rows above it are bad-state rows)
    tables: dict = dataclasses.field(default_factory=dict)  # block tables (read-only)

    @property
    def B(self):
        return self.topk.shape[0]

    def copy(self) -> "Case":
        return dataclasses.replace(self, **{
            f.name: (getattr(self, f.name).copy() if isinstance(getattr(self, f.name), np.ndarray)
                     else getattr(self, f.name)) for f in dataclasses.fields(self)})


def random_case(rng, *, B, K, H, S, R=None, seq_len=None, P=None, cols=None, with_v=False,
                permuted_rows=True, extra_hot=3, width_pad=0) -> Case:
    R = R if R is not None else B + 1
    seq_len = seq_len if seq_len is not None else max(H + 1, 3 * H)
    cols = cols if cols is not None else int(np.max(seq_len))
    P = P if P is not None else R * cols
    tokens, rows, lru = synth.cold_state(R, H, width=H + 1 + width_pad,
                                         seed=int(rng.integers(1 << 30)) if permuted_rows else None)
    hot_rows = R * (H + 1) + extra_hot
    pool_rows = np.stack([rng.permutation(P)[:cols] for _ in range(R)]).astype(np.int64)
    pool_k = rng.integers(0, 256, size=(P, S), dtype=np.uint8)
    pool_v = rng.integers(0, 256, size=(P, S), dtype=np.uint8) if with_v else None
    hot_k = rng.integers(0, 256, size=(hot_rows, S), dtype=np.uint8)
    hot_v = rng.integers(0, 256, size=(hot_rows, S), dtype=np.uint8) if with_v else None
    req_state = rng.permutation(R)[:B].astype(np.int64)
    seq_lens = np.broadcast_to(np.asarray(seq_len, dtype=np.int64), (B,)).copy()
    topk = np.zeros((B, K), dtype=np.int32)
    return Case(H, K, S, topk, seq_lens, req_state, tokens, rows, lru, pool_rows, pool_k,
                pool_v, hot_k, hot_v)


def random_ids(rng, case: Case, *, p_invalid=0.1, p_dup=0.1, p_newest=0.1, p_reuse=0.5,
               prev=None) -> np.ndarray:
    """Random top-k rows with invalid, duplicate, newest and reused ids mixed in."""
    out = np.zeros((case.B, case.K), dtype=np.int32)
    for b in range(case.B):
        L = int(case.seq_lens[b])
        row = []
        for i in range(case.K):
            u = rng.random()
            if u < p_invalid:
                row.append(int(rng.choice([-1, -7, L, L + 3])))
            elif u < p_invalid + p_dup and row:
                row.append(int(rng.choice(row)))
            elif u < p_invalid + p_dup + p_newest:
                row.append(L - 1)
            elif prev is not None and u < p_invalid + p_dup + p_newest + p_reuse:
                row.append(int(rng.choice(prev[b])))
            else:
                row.append(int(rng.integers(0, max(1, L))))
        out[b] = row
    return out


PLAN_FILL_SRC, PLAN_FILL_DST = 3, 1  # valid-looking values in unwritten plan entries


def run_oracle(case: Case, mutant: int = 0, plan: bool = False):
    """One oracle step; mutates ``case`` state, returns (out, miss, status, stats),
    plus (miss_src, miss_dst, miss_mask) when ``plan``."""
    import oracle

    out = np.full((case.B, case.K), 12345, dtype=np.int32)
    miss = np.full(case.B, 777, dtype=np.int32)
    status = np.full(case.B, 999, dtype=np.int32)
    stats = np.zeros(2, dtype=np.uint64)
    kw = {}
    if plan:
        kw = dict(miss_src=np.full((case.B, case.K), PLAN_FILL_SRC, dtype=np.int64),
                  miss_dst=np.full((case.B, case.K), PLAN_FILL_DST, dtype=np.int32),
                  miss_mask=np.full((case.B, case.K), 7, dtype=np.int32))
    oracle.swap_in(topk_ids=case.topk, seq_lens=case.seq_lens, req_state=case.req_state,
                   slot_tokens=case.tokens, slot_rows=case.rows, lru=case.lru,
                   pool_rows=case.pool_rows, pool_k=case.pool_k, pool_v=case.pool_v,
                   hot_k=case.hot_k, hot_v=case.hot_v, out_rows=out, hot_size=case.H,
                   num_real=case.num_real, miss_count=miss, stats=stats, status=status,
                   mutant=mutant, max_seq_len=case.max_seq_len, **kw, **case.tables)
    if plan:
        return out, miss, status, stats, kw["miss_src"], kw["miss_dst"], kw["miss_mask"]
    return out, miss, status, stats


def run_brute(case: Case, plans=None):
    """One brute-force step on list copies; writes the new state back into ``case``.
    When ``plans`` is a list it receives one miss-plan dict per batch row."""
    import brute

    H = case.H
    state = {"tokens": [list(map(int, r)) for r in case.tokens],
             "rows": [list(map(int, r)) for r in case.rows],
             "lru": [list(map(int, r[:H])) for r in case.lru]}
    pool_rows = [list(map(int, r)) for r in case.pool_rows]
    pool = [bytes(r) for r in case.pool_k]
    hot = [bytearray(r) for r in case.hot_k]
    assert case.pool_v is None, "brute force models K rows only"
    outs, miss, status, stats = brute.swap_in(
        [list(map(int, r)) for r in case.topk], [int(x) for x in case.seq_lens],
        [int(x) for x in case.req_state], H, state, pool_rows, pool, hot,
        num_real=case.num_real, plans=plans)
    case.tokens[:] = np.array(state["tokens"], dtype=np.int32)
    case.lru[:, :H] = np.array(state["lru"], dtype=np.int16)
    case.hot_k[:] = np.frombuffer(b"".join(bytes(r) for r in hot), dtype=np.uint8).reshape(
        case.hot_k.shape)
    return (np.array(outs, dtype=np.int32).reshape(case.B, case.K),
            np.array(miss, dtype=np.int32), np.array(status, dtype=np.int32),
            np.array(stats, dtype=np.uint64))


def assert_same_state(a: Case, b: Case, what=""):
    np.testing.assert_array_equal(a.tokens, b.tokens, err_msg=f"slot_tokens {what}")
    np.testing.assert_array_equal(a.lru, b.lru, err_msg=f"lru {what}")
    np.testing.assert_array_equal(a.hot_k, b.hot_k, err_msg=f"hot_k {what}")
    if a.hot_v is not None or b.hot_v is not None:
        np.testing.assert_array_equal(a.hot_v, b.hot_v, err_msg=f"hot_v {what}")


def corrupt(rng, case: Case, kinds=("lru_range", "lru_dup", "pool_row", "hot_row", "state")):
    """Inject host-side corruption into long-lived state (never on the device)."""
    R, H = case.lru.shape[0], case.H
    for k in kinds:
        if rng.random() < 0.5:
            continue
        r = int(rng.integers(R))
        if k == "lru_range":
            case.lru[r, int(rng.integers(H))] = int(rng.choice([-1, H, H + 5, 32767]))
        elif k == "lru_dup" and H > 1:
            p, q = rng.choice(H, size=2, replace=False)
            case.lru[r, p] = case.lru[r, q]
        elif k == "pool_row":
            c = int(rng.integers(case.pool_rows.shape[1]))
            case.pool_rows[r, c] = int(rng.choice([-1, case.pool_k.shape[0],
                                                   case.pool_k.shape[0] + 9]))
        elif k == "hot_row":
            case.rows[r, int(rng.integers(H))] = int(rng.choice([-1, case.hot_k.shape[0],
                                                                 1 << 30]))
        elif k == "state" and case.B > 0:
            case.req_state[int(rng.integers(case.B))] = int(rng.choice([-1, R, R + 4]))


def oracle_st_bad_state():
    import oracle
    return oracle.ST_BAD_STATE
