"""Brute-force restatement of the swap-in for tiny inputs (pure Python lists).

Independent of the C++ oracle: no hash maps or sets, only O(H*K) list scans,
and the LRU writeback is computed three ways -- as the plain concatenation
[stale evictables][misses, top-k order][hits, old order], with the index
formula of SGLang jit_kernel/csrc/hisparse.cuh (load_cache_to_device_buffer_kernel,
"Write back LRU order" block), and with the index formula of vLLM
csrc/libtorch_stable/hisparse_kernels.cu (hisparse_resolve_residency_kernel,
"Phase 4") -- and the three are asserted equal on every call.

Used only by the tests.
"""
from __future__ import annotations

DUP, BAD_POOL, BAD_LRU, BAD_HOT, TIMEOUT, BAD_STATE = 1, 2, 4, 8, 16, 32


def writeback_concat(hits, evict, M):
    return [s for s, _ in evict[M:]] + [s for s, _ in evict[:M]] + list(hits)


def _compacted(hits, evict, H):
    # hits forward from index 0, evictables backward from H-1 (the pages'
    # compacted slot buffer)
    buf = [None] * H
    for j, s in enumerate(hits):
        buf[j] = s
    for e, (s, _) in enumerate(evict):
        buf[H - 1 - e] = s
    return buf


def writeback_sglang(hits, evict, M, H):
    buf = _compacted(hits, evict, H)
    E = H - len(hits)
    new = [None] * H
    for i in range(H):
        if i < M:
            new[E - M + i] = buf[H - 1 - i]
        elif i < E:
            new[i - M] = buf[H - 1 - i]
        else:
            new[i] = buf[i - E]
    return new


def writeback_vllm(hits, evict, M, H):
    buf = _compacted(hits, evict, H)
    E = H - len(hits)
    remaining = E - M
    new = [None] * H
    for i in range(H):
        if i < remaining:
            new[i] = buf[H - 1 - M - i]
        elif i < remaining + M:
            new[i] = buf[H - 1 - (i - remaining)]
        else:
            new[i] = buf[i - remaining - M]
    return new


def swap_in_row(ids, seq_len, H, tokens, rows, lru, pool_rows, pool, hot, hot_num_rows,
                plan=None):
    """One batch row.  ``tokens``/``rows`` are lists of length >= H+1, ``lru`` a list
    of length H, ``pool_rows`` a list (token -> pool row), ``pool`` a list of bytes
    rows, ``hot`` a list of bytearray rows.  Mutates tokens, lru, hot.
    Returns (out, miss_count, hits, status).  When ``plan`` is a dict it receives
    the miss plan: 'src' (pool row of each miss, in order), 'dst' (the hot row it
    was given, or -1) and 'mask' (1 for each top-k entry that was a miss)."""
    K = len(ids)
    out = [-1] * K
    if plan is not None:
        plan.update(src=[], dst=[], mask=[0] * K)
    if seq_len <= H:
        count = min(seq_len, K)
        for i in range(K):
            t = ids[i]
            if i < count and 0 <= t < seq_len:
                out[i] = rows[t]
        return out, 0, 0, 0

    st = 0
    kind = ["invalid"] * K
    for i in range(K):
        t = ids[i]
        if not (0 <= t < seq_len):
            continue
        if any(ids[j] == t for j in range(i)):
            kind[i] = "dup"
            st |= DUP
            continue
        if t == seq_len - 1:
            kind[i] = "newest"
            out[i] = rows[H]
            continue
        kind[i] = "want"

    resolved = [False] * K
    hits, evict = [], []
    for p in range(H):
        s = lru[p]
        if not (0 <= s < H) or s in lru[:p]:
            st |= BAD_LRU
            evict.append((s, True))
            continue
        tok = tokens[s]
        hit_i = None
        for i in range(K):
            if kind[i] == "want" and ids[i] == tok and not resolved[i]:
                hit_i = i
                break
        if hit_i is None:
            evict.append((s, False))
        else:
            resolved[hit_i] = True
            out[hit_i] = rows[s]
            hits.append(s)

    misses = []
    for i in range(K):
        if kind[i] != "want" or resolved[i]:
            continue
        t = ids[i]
        pr = pool_rows[t] if t < len(pool_rows) else -1
        if not (0 <= pr < len(pool)):
            st |= BAD_POOL
            continue
        misses.append((i, t, pr))
    M = len(misses)
    assert M <= len(evict)

    for m, (i, t, pr) in enumerate(misses):
        if plan is not None:
            plan["mask"][i] = 1
            plan["src"].append(pr)
            plan["dst"].append(-1)
        s, bad = evict[m]
        if bad:
            st |= BAD_LRU
            continue
        hr = rows[s]
        if not (0 <= hr < hot_num_rows):
            st |= BAD_HOT
            continue
        if plan is not None:
            plan["dst"][m] = hr
        out[i] = hr
        tokens[s] = t
        hot[hr][:] = pool[pr]

    a = writeback_concat(hits, evict, M)
    b = writeback_sglang(hits, evict, M, H)
    c = writeback_vllm(hits, evict, M, H)
    assert a == b == c, (a, b, c)
    lru[:] = a
    return out, M, len(hits), st


def swap_in(ids_rows, seq_lens, req_state, H, state, pool_rows, pool, hot, num_real=-1,
            plans=None):
    """Batch version over dict-of-lists state {'tokens','rows','lru'} keyed by state row.
    When ``plans`` is a list, one miss-plan dict per batch row is appended to it."""
    outs, miss, status = [], [], []
    stats = [0, 0]
    for b, ids in enumerate(ids_rows):
        plan = {"src": [], "dst": [], "mask": [0] * len(ids)}
        if plans is not None:
            plans.append(plan)
        r = req_state[b]
        if (num_real >= 0 and b >= num_real) or r < 0:
            outs.append([-1] * len(ids)); miss.append(0); status.append(0)
            continue
        if r >= len(state["tokens"]):
            outs.append([-1] * len(ids)); miss.append(0); status.append(BAD_STATE)
            continue
        o, m, h, st = swap_in_row(list(ids), seq_lens[b], H, state["tokens"][r],
                                  state["rows"][r], state["lru"][r], pool_rows[r], pool, hot,
                                  len(hot), plan=plan)
        outs.append(o); miss.append(m); status.append(st)
        if seq_lens[b] > H:
            stats[0] += h
            stats[1] += m
    return outs, miss, status, stats


def gather_misses(plans, miss_count, pool, hot):
    """Replay per-row miss plans onto another layer's pool/hot rows (lists)."""
    status = 0
    for b, plan in enumerate(plans):
        for m in range(max(0, min(miss_count[b], len(plan["mask"])))):
            s, d = plan["src"][m], plan["dst"][m]
            if d < 0:
                continue
            if not (0 <= s < len(pool)) or d >= len(hot):
                status |= 64
                continue
            hot[d][:] = pool[s]
    return status
