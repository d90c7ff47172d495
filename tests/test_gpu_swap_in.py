"""GPU parity for hs_swap_in: bit-exact against the CPU oracle (indices, LRU
state, slot tokens, hot-buffer bytes, counters and status bits), through the
C ABI, over tiny exhaustive-style cases, ragged multi-tile sizes, every copy
width (16-byte, 4-byte, byte), K+V, pinned-host pools, int32/int64 index
types, padding rows and host-injected corruption."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import cases
from gpu_cases import GpuCase, step_both

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__

    __graft_entry__.build()
    return torch.device("cuda:0")


def test_golden_worked_example_on_gpu(dev):
    import json
    import os

    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                    "swap_in_worked_example.json")))
    H, L = g["hot_size"], g["seq_len"]
    W = H + 1
    c = cases.Case(H=H, K=3, S=2, topk=np.zeros((1, 3), np.int32),
                   seq_lens=np.array([L], np.int64), req_state=np.zeros(1, np.int64),
                   tokens=np.full((1, W), -1, np.int32),
                   rows=np.array([g["slot_rows"]], np.int32),
                   lru=np.arange(H, dtype=np.int16)[None], pool_rows=
                   np.array([[50 + t for t in range(L)]], np.int64),
                   pool_k=np.array([[x % 256, (x + 1) % 256] for x in range(64)], np.uint8),
                   pool_v=None, hot_k=np.full((105, 2), 0xEE, np.uint8), hot_v=None)
    gc = GpuCase(c.copy(), dev)
    for st in g["steps"]:
        out, miss, status, _ = gc.step(np.array([st["ids"]], np.int32))
        assert out[0].tolist() == st["out"]
        assert int(miss[0]) == st["miss_count"] and int(status[0]) == st["status"]
        assert gc.lru.cpu().numpy()[0].tolist() == st["lru"]


@pytest.mark.parametrize("seed", range(40))
def test_random_tiny_with_corruption(dev, seed):
    rng = np.random.default_rng(5000 + seed)
    H = int(rng.integers(1, 40))
    K = int(rng.integers(1, H + 1))
    B = int(rng.integers(1, 6))
    S = int(rng.choice([1, 3, 4, 16, 17, 132, 656]))
    seq = rng.integers(1, 4 * H + 3, size=B)
    ref = cases.random_case(rng, B=B, K=K, H=H, S=S, R=B + 2, seq_len=seq,
                            P=int(rng.integers(4 * H + 3, 8 * H + 8)),
                            with_v=bool(seed % 3 == 0))
    ref.num_real = int(rng.choice([-1, B, max(0, B - 1)]))
    g = GpuCase(ref.copy(), dev, pool_in_host=bool(seed % 4 == 1),
                seq_dtype=torch.int32 if seed % 2 else torch.int64,
                req_dtype=torch.int32 if seed % 5 == 0 else torch.int64)
    g.case = ref
    prev = None
    for step in range(6):
        ids = cases.random_ids(rng, ref, prev=prev)
        prev = ids
        if step >= 3:
            cases.corrupt(np.random.default_rng(seed * 7 + step), ref)
            g.push_state(ref)
        step_both(g, ref, ids, f"seed={seed} step={step}", plan=seed % 2 == 0)


@pytest.mark.parametrize("H,K,S,B,with_v,host", [
    (1000, 700, 656, 5, False, False),     # several 1024-thread tiles, ragged tail
    (2500, 2500, 132, 3, False, True),     # K == H, 4-byte path, pinned host pool
    (4096, 2048, 656, 4, True, False),     # K and V
    (3001, 1237, 17, 2, False, False),     # byte path, odd sizes
    (777, 33, 2048, 3, False, True),
])
def test_multi_tile_workloads(dev, H, K, S, B, with_v, host):
    rng = np.random.default_rng(H * 7 + K)
    L = 8 * H
    ref = cases.random_case(rng, B=B, K=K, H=H, S=S, R=B + 1, seq_len=L, with_v=with_v,
                            width_pad=3)
    g = GpuCase(ref.copy(), dev, pool_in_host=host)
    g.case = ref
    import synth
    ts = synth.TopkStream(H, 0, B, K, L, 0.6)
    for step in range(5):
        step_both(g, ref, ts.next(), f"H={H} step={step}", plan=True)
    # a step with invalid, duplicate and newest ids mixed in
    step_both(g, ref, cases.random_ids(rng, ref), "mixed", plan=True)


def test_all_rows_padding_and_empty(dev):
    rng = np.random.default_rng(3)
    ref = cases.random_case(rng, B=3, K=8, H=16, S=16, R=4, seq_len=50)
    ref.num_real = 0
    g = GpuCase(ref.copy(), dev)
    g.case = ref
    out, miss, status, stats = step_both(g, ref, cases.random_ids(rng, ref), "num_real=0")
    assert np.all(out == -1) and np.all(miss == 0)


def test_capture_in_cuda_graph(dev):
    """A swap-in captured in a CUDA graph and replayed matches eager calls."""
    import sparse_attention_kv_row_gb300 as hs
    import synth

    rng = np.random.default_rng(9)
    H, K, B, L = 256, 64, 4, 4000
    ref = cases.random_case(rng, B=B, K=K, H=H, S=656, R=B, seq_len=L)
    g = GpuCase(ref.copy(), dev)
    ts = synth.TopkStream(1, 0, B, K, L, 0.5)
    topk = torch.zeros((B, K), dtype=torch.int32, device=dev)
    out = torch.zeros((B, K), dtype=torch.int32, device=dev)
    seq = torch.from_numpy(ref.seq_lens).to(dev)
    req = torch.from_numpy(ref.req_state).to(dev)
    args = hs.make_swap_in_args(topk_ids=topk, seq_lens=seq, req_state=req,
                                slot_tokens=g.tokens, slot_rows=g.rows, lru=g.lru,
                                pool_rows=g.pool_rows, pool_k=g.pool_k, hot_k=g.hot_k,
                                out_rows=out)
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    # one eager call first (one-time kernel set-up), then restore the state
    snap = (g.tokens.clone(), g.lru.clone(), g.hot_k.clone())
    with torch.cuda.stream(s):
        hs.swap_in_args(args, stream=s)
    torch.cuda.synchronize()
    g.tokens.copy_(snap[0]); g.lru.copy_(snap[1]); g.hot_k.copy_(snap[2])
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=s):
        hs.swap_in_args(args, stream=s)
    torch.cuda.synchronize()
    for step in range(4):
        ids = ts.next()
        topk.copy_(torch.from_numpy(ids))
        graph.replay()
        torch.cuda.synchronize()
        ref.topk = ids
        r_out, _, _, _ = cases.run_oracle(ref)
        np.testing.assert_array_equal(out.cpu().numpy(), r_out)
        g.assert_matches(ref, f"graph step {step}")


def test_row_subsets_match_whole_batch(dev):
    """Rows are independent: two disjoint halves of the batch, swapped in by two
    calls (as two GPUs of a data-parallel job would), give exactly the results
    of one whole-batch call."""
    import sparse_attention_kv_row_gb300 as hs
    import synth

    rng = np.random.default_rng(77)
    B, K, H, L = 6, 96, 256, 3000
    base = cases.random_case(rng, B=B, K=K, H=H, S=656, R=B, seq_len=L)
    whole = GpuCase(base.copy(), dev)
    split = GpuCase(base.copy(), dev)
    ts = synth.TopkStream(3, 0, B, K, L, 0.7)
    for step in range(4):
        ids = ts.next()
        whole_out = whole.step(ids)[0]
        split_out = []
        for rows_ in (slice(0, 3), slice(3, 6)):
            sub = torch.from_numpy(np.ascontiguousarray(ids[rows_])).to(dev)
            out = torch.empty((3, K), dtype=torch.int32, device=dev)
            hs.swap_in(topk_ids=sub,
                       seq_lens=torch.from_numpy(base.seq_lens[rows_]).to(dev),
                       req_state=torch.from_numpy(base.req_state[rows_]).to(dev),
                       slot_tokens=split.tokens, slot_rows=split.rows, lru=split.lru,
                       pool_rows=split.pool_rows, pool_k=split.pool_k, hot_k=split.hot_k,
                       out_rows=out)
            split_out.append(out)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(whole_out, torch.cat(split_out).cpu().numpy())
        for a, b in ((whole.tokens, split.tokens), (whole.lru, split.lru),
                     (whole.hot_k, split.hot_k)):
            assert torch.equal(a, b), f"step {step}"


@pytest.mark.parametrize("mode,shape", [("chain", "small"), ("interleaved", "small"),
                                        ("graph", "small"), ("chain", "clusters")])
def test_overlap_prev(dev, mode, shape):
    """HS_OVERLAP_PREV: launches that may start before the preceding kernel
    finishes still match the oracle.  'chain': one kernel writes every layer's
    top-k rows, then the layers' swap-ins run back to back (each may overlap
    the one before); 'interleaved': a kernel writes layer l's top-k rows right
    before layer l's swap-in; 'graph': the chain captured in a CUDA graph.
    Rows include a padding row and a short sequence (the fast path).  'small'
    has no sequence bound (the wide request hash); 'clusters' is the decode
    shape (32 rows, top-k 2048, hot size 4096: 128 CTAs, so part of each launch
    starts while the previous one runs) with the bound given (the packed hash),
    and every row's status must be clean."""
    import sparse_attention_kv_row_gb300 as hs
    import synth

    rng = np.random.default_rng(123)
    if shape == "small":
        NL, B, K, H, L, bound = 4, 5, 300, 1000, 9000, 0
    else:
        NL, B, K, H, L, bound = 3, 32, 2048, 4096, 20000, 20000
    refs, gpus = [], []
    for l in range(NL):
        ref = cases.random_case(rng, B=B, K=K, H=H, S=132 if shape == "small" else 16,
                                R=B + 2, seq_len=L)
        ref.seq_lens[1] = H - 3  # fast path
        ref.num_real = B - 1     # last row is padding
        refs.append(ref)
        gpus.append(GpuCase(ref.copy(), dev))
    stream_ = [synth.TopkStream(40 + l, 0, B, K, L, 0.8) for l in range(NL)]
    # top-k rows sit at the end of a large buffer so the writing kernel reaches them late
    big = 1 << 24
    src = torch.zeros(big + NL * B * K, dtype=torch.int32, device=dev)
    dst = torch.zeros_like(src)
    topk = dst[big:].view(NL, B, K)
    outs = torch.zeros((NL, B, K), dtype=torch.int32, device=dev)
    miss = torch.zeros((NL, B), dtype=torch.int32, device=dev)
    status = torch.zeros((NL, B), dtype=torch.int32, device=dev)
    num_real = torch.tensor([B - 1], dtype=torch.int32, device=dev)
    args = [hs.make_swap_in_args(
        topk_ids=topk[l], seq_lens=torch.from_numpy(refs[l].seq_lens).to(dev),
        req_state=torch.from_numpy(refs[l].req_state).to(dev), slot_tokens=gpus[l].tokens,
        slot_rows=gpus[l].rows, lru=gpus[l].lru, pool_rows=gpus[l].pool_rows,
        pool_k=gpus[l].pool_k, hot_k=gpus[l].hot_k, out_rows=outs[l], miss_count=miss[l],
        num_real=num_real, overlap_prev=True, status=status[l], max_seq_len=bound)
        for l in range(NL)]
    s = torch.cuda.Stream()

    def step_chain():
        torch.add(src, 0, out=dst)
        for a in args:
            hs.swap_in_args(a, stream=s)

    graph = None
    if mode == "graph":
        snap = [(g.tokens.clone(), g.lru.clone(), g.hot_k.clone()) for g in gpus]
        with torch.cuda.stream(s):
            step_chain()  # one eager pass first (one-time kernel set-up), then restore
        torch.cuda.synchronize()
        for g, (t, lr, hk) in zip(gpus, snap):
            g.tokens.copy_(t); g.lru.copy_(lr); g.hot_k.copy_(hk)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            step_chain()
        torch.cuda.synchronize()
    for step in range(4):
        ids = np.stack([st.next() for st in stream_])
        src[big:].copy_(torch.from_numpy(ids.reshape(-1)))
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            if mode == "chain":
                step_chain()
            elif mode == "interleaved":
                for l in range(NL):
                    torch.add(src[big + l * B * K: big + (l + 1) * B * K], l * 0,
                              out=dst[big + l * B * K: big + (l + 1) * B * K])
                    hs.swap_in_args(args[l], stream=s)
            else:
                graph.replay()
        torch.cuda.synchronize()
        for l in range(NL):
            refs[l].topk = ids[l]
            r_out, r_miss, _, _ = cases.run_oracle(refs[l])
            np.testing.assert_array_equal(outs[l].cpu().numpy(), r_out, f"{mode} {step} {l}")
            np.testing.assert_array_equal(miss[l].cpu().numpy(), r_miss)
            gpus[l].assert_matches(refs[l], f"{mode} step {step} layer {l}")
        if shape == "clusters":
            assert int(status.abs().max()) == 0, status.cpu().numpy()


def test_wide_hash_long_sequences(dev):
    """Ids beyond 2^(32 - entry bits) - 1 (here K=2100, so ids >= 2^20 - 1) take the wide
    {id, entry} form of the request hash; the results match the oracle all the same."""
    rng = np.random.default_rng(2024)
    B, K, H, L = 2, 2100, 2300, 1_200_000
    ref = cases.random_case(rng, B=B, K=K, H=H, S=16, R=B + 1, seq_len=L)
    ref.seq_lens[1] = 600_000   # this row stays in the packed form
    g = GpuCase(ref.copy(), dev, seq_bound=0)   # no bound given: the wide form
    g.case = ref
    import synth
    ts = synth.TopkStream(77, 0, B, K, 600_000, 0.7)
    for step in range(4):
        ids = ts.next().copy()
        ids[0] += rng.integers(0, 2, K, dtype=np.int32) * 590_000   # row 0: ids up to ~1.19M
        step_both(g, ref, ids, f"step {step}", plan=True)
    step_both(g, ref, cases.random_ids(rng, ref), "mixed", plan=True)


def test_sequence_bound(dev):
    """Rows longer than the caller's max_seq_len are bad-state rows on both sides;
    the others are resolved with the compact hash."""
    rng = np.random.default_rng(31)
    ref = cases.random_case(rng, B=4, K=64, H=200, S=16, R=5, seq_len=2000)
    ref.seq_lens[2] = 2500
    ref.max_seq_len = 2200
    g = GpuCase(ref.copy(), dev)
    g.case = ref
    prev = None
    for step in range(3):
        ids = cases.random_ids(rng, ref, prev=prev)
        prev = ids
        res = step_both(g, ref, ids, f"step {step}", plan=True)
        out, status = res[0], res[2]
        assert status[2] == cases.oracle_st_bad_state() and np.all(out[2] == -1)


def test_bounded_wait_runs_out_and_context_stays_usable(dev):
    """A wait that runs out hands control back with HS_ST_TIMEOUT: the library's
    bounded mbarrier wait on a barrier that nothing arms (no copy in flight).
    The swap-ins that follow on the same context still match the oracle."""
    import oracle
    import sparse_attention_kv_row_gb300 as hs

    st = torch.zeros(1, dtype=torch.int32, device=dev)
    hs.wait_selftest(1000, st)
    torch.cuda.synchronize()
    assert st.item() == oracle.ST_TIMEOUT
    rng = np.random.default_rng(31)
    ref = cases.random_case(rng, B=3, K=40, H=100, S=32)
    g = GpuCase(ref.copy(), dev)
    prev = None
    for step in range(3):
        ids = cases.random_ids(rng, ref, prev=prev)
        prev = ids
        step_both(g, ref, ids, f"after the timeout, step {step}")


@pytest.mark.parametrize("which,rank,overlap", [(0, 0, False), (0, -1, False), (1, -1, False),
                                                (1, 3, True), (0, 2, True)])
def test_forced_timeout_leaves_rows_alone(dev, which, rank, overlap):
    """One CTA of every full-path row gives up a bounded wait at once (the
    self-test entry point; the copy it gave up on is still waited out, so
    nothing faults or hangs).  The whole row is then left alone, whichever CTA
    of the cluster gave up: status is exactly HS_ST_TIMEOUT, miss_count 0, and
    the outputs, plan, LRU order, slot tokens, statistics and hot buffer are
    unchanged.  A padding row and a short-sequence row do not wait and come
    out as the oracle says.  A normal call afterwards matches the oracle."""
    import oracle
    import sparse_attention_kv_row_gb300 as hs
    import synth

    rng = np.random.default_rng(600 + which * 10 + rank)
    B, K, H, L = 5, 300, 1000, 9000      # 5 rows: clusters of 8 CTAs
    ref = cases.random_case(rng, B=B, K=K, H=H, S=656, R=B + 1, seq_len=L)
    ref.seq_lens[1] = H - 5              # the short-sequence path
    ref.req_state[3] = -1                # padding
    g = GpuCase(ref.copy(), dev)
    ts = synth.TopkStream(5, 0, B, K, L, 0.6)
    step_both(g, ref, ts.next(), "warm")           # some resident tokens first
    ids = ts.next()
    before = (g.tokens.clone(), g.lru.clone(), g.hot_k.clone())
    topk = torch.from_numpy(ids).to(dev)
    out = torch.full((B, K), 4242, dtype=torch.int32, device=dev)
    miss = torch.full((B,), 777, dtype=torch.int32, device=dev)
    status = torch.full((B,), 999, dtype=torch.int32, device=dev)
    stats = torch.zeros(2, dtype=torch.int64, device=dev)
    plan_src = torch.full((B, K), 5, dtype=torch.int64, device=dev)
    plan_dst = torch.full((B, K), 6, dtype=torch.int32, device=dev)
    mask = torch.full((B, K), 7, dtype=torch.int32, device=dev)
    args = hs.make_swap_in_args(
        topk_ids=topk, seq_lens=torch.from_numpy(ref.seq_lens).to(dev),
        req_state=torch.from_numpy(ref.req_state).to(dev), slot_tokens=g.tokens,
        slot_rows=g.rows, lru=g.lru, pool_rows=g.pool_rows, pool_k=g.pool_k, hot_k=g.hot_k,
        out_rows=out, miss_count=miss, status=status, stats=stats, miss_src=plan_src,
        miss_dst=plan_dst, miss_mask=mask, max_seq_len=L, overlap_prev=overlap)
    hs.swap_in_timeout_selftest(args, rank=rank, which=which)
    torch.cuda.synchronize()
    assert torch.equal(g.tokens, before[0]) and torch.equal(g.lru, before[1])
    assert torch.equal(g.hot_k, before[2])
    assert int(stats.abs().sum()) == 0
    full = [0, 2, 4]
    st, ms, o = status.cpu().numpy(), miss.cpu().numpy(), out.cpu().numpy()
    for b in full:
        assert st[b] == oracle.ST_TIMEOUT and ms[b] == 0, (b, st, ms)
        assert np.all(o[b] == 4242)
        assert np.all(plan_src[b].cpu().numpy() == 5) and np.all(mask[b].cpu().numpy() == 7)
    # the rows that do not wait: as the oracle has them (their state is untouched)
    probe = ref.copy()
    probe.topk = ids
    r_out, r_miss, r_status, _ = cases.run_oracle(probe)
    for b in (1, 3):
        np.testing.assert_array_equal(o[b], r_out[b])
        assert ms[b] == r_miss[b] and st[b] == r_status[b]
    # the context is usable and the state intact: a normal call matches the oracle
    step_both(g, ref, ids, "after the forced time-out", plan=True)


@pytest.mark.parametrize("layers_api", [False, True])
def test_packed_hash_when_the_bound_is_too_long_for_the_direct_map(dev, layers_api):
    """A sequence bound above 2^24 rules out the layers kernel's direct request
    map; with top_k 64 the packed hash still fits every id (the per-layer
    kernel's hash too).  Results match the oracle all the same."""
    import sparse_attention_kv_row_gb300 as hs
    import synth

    rng = np.random.default_rng(4242)
    B, K, H, L = 3, 64, 300, 5000
    ref = cases.random_case(rng, B=B, K=K, H=H, S=656, R=B + 1, seq_len=L)
    g = GpuCase(ref.copy(), dev, seq_bound=30_000_000)
    g.case = ref
    ts = synth.TopkStream(21, 0, B, K, L, 0.6)
    for step in range(4):
        ids = ts.next() if step < 3 else cases.random_ids(rng, ref)
        if not layers_api:
            step_both(g, ref, ids, f"step {step}", plan=True)
            continue
        out = torch.full((B, K), 12345, dtype=torch.int32, device=dev)
        miss = torch.zeros(B, dtype=torch.int32, device=dev)
        status = torch.zeros(B, dtype=torch.int32, device=dev)
        a = hs.make_swap_in_args(
            topk_ids=torch.from_numpy(ids).to(dev), seq_lens=torch.from_numpy(ref.seq_lens).to(dev),
            req_state=torch.from_numpy(ref.req_state).to(dev), slot_tokens=g.tokens,
            slot_rows=g.rows, lru=g.lru, pool_rows=g.pool_rows, pool_k=g.pool_k, hot_k=g.hot_k,
            out_rows=out, miss_count=miss, status=status, max_seq_len=30_000_000)
        hs.swap_in_layers([a])
        torch.cuda.synchronize()
        ref.topk = ids
        r_out, r_miss, r_status, _ = cases.run_oracle(ref)
        np.testing.assert_array_equal(out.cpu().numpy(), r_out)
        np.testing.assert_array_equal(miss.cpu().numpy(), r_miss)
        np.testing.assert_array_equal(status.cpu().numpy(), r_status)
        g.assert_matches(ref, f"layers step {step}")
