"""GPU parity for the miss plan and its replay (hs_gather_misses), through the
C ABI, against the CPU oracle element by element:

- random plans with no-row misses, bad pool rows, bad hot rows and counts
  outside [0, top_k], K-only and K+V, HBM and pinned-host pools, 16-byte,
  4-byte and byte rows;
- the replay identity on the GPU: a resolving layer's plan replayed onto a
  second layer with the same state gives that layer's own resolution, over
  several steps and with the layers captured as one CUDA graph;
- empty calls launch nothing.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import cases
import oracle
from gpu_cases import GpuCase

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__

    __graft_entry__.build()
    return torch.device("cuda:0")


def _hs():
    import sparse_attention_kv_row_gb300 as hs

    return hs


@pytest.mark.parametrize("S,with_v,host,NL,B", [(656, False, False, 1, 6), (656, True, True, 3, 6),
                                                 (132, True, False, 2, 6), (17, False, True, 3, 6),
                                                 (656, True, False, 4, 160),
                                                 (132, True, False, 4, 160)])
def test_gather_matches_oracle(dev, S, with_v, host, NL, B):
    """NL layers (K, then V when with_v) replayed by one call; the oracle
    replays layer by layer.  With B=160 rows a block holds about 40 misses x 8
    pointer pairs, more than one round of staged units (16-byte path at 656 B
    rows, one warp per unit at 132 B)."""
    rng = np.random.default_rng(S * 3 + with_v + B)
    K, P = (300, 5000) if B == 6 else (120, 3000)
    R = 2000 if B == 6 else B * K + 500
    NP = NL * (2 if with_v else 1)
    pools = [rng.integers(0, 256, (P, S), dtype=np.uint8) for _ in range(NP)]
    hots = [rng.integers(0, 256, (R, S), dtype=np.uint8) for _ in range(NP)]
    src = rng.integers(0, P, (B, K)).astype(np.int64)
    # distinct destinations across the whole call (the documented precondition)
    dst = rng.choice(R, size=B * K, replace=False).astype(np.int32).reshape(B, K)
    src[0, 3], dst[1, 5], dst[2, 7] = P + 2, R + 1, -1   # bad src, bad dst, no row
    src[3, 0] = -4
    count = np.array([K, 0, 17, -3, K + 50, 250], np.int32)
    if B > 6:
        count = np.concatenate([count, np.full(B - 6, K, np.int32)])
    st_ref = np.zeros(1, np.int32)
    refs = [h.copy() for h in hots]
    for pl, hr in zip(pools, refs):
        oracle.gather_misses(pool_k=pl, hot_k=hr, miss_src=src, miss_dst=dst, miss_count=count,
                             status=st_ref)

    def put(a, pinned=False):
        if a is None:
            return None
        t = torch.from_numpy(a.copy())
        return t.pin_memory() if pinned else t.to(dev)

    g_hot = [put(h) for h in hots]
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    _hs().gather_misses([put(pl, host) for pl in pools], g_hot, put(src), put(dst), put(count),
                        has_v=with_v, status=st)
    torch.cuda.synchronize()
    for n, (g, hr) in enumerate(zip(g_hot, refs)):
        np.testing.assert_array_equal(g.cpu().numpy(), hr, err_msg=f"layer {n}")
    assert st.item() == st_ref[0] == oracle.ST_BAD_INDEX


@pytest.mark.parametrize("with_v", [False, True])
@pytest.mark.parametrize("overlap", [False, True])
def test_replay_equals_resolution_on_gpu(dev, with_v, overlap):
    """Layer A resolves and emits its plan; layer B (same state, other bytes)
    replays it; layer C (a copy of B) resolves itself.  B and C must agree.
    With overlap the replay and C's swap-in are launched with HS_OVERLAP_PREV
    (each may start while the kernel before it runs)."""
    import synth

    hs = _hs()
    rng = np.random.default_rng(55 + with_v)
    B, K, H, L, S = 5, 400, 1100, 9000, 656
    A = cases.random_case(rng, B=B, K=K, H=H, S=S, R=B + 1, seq_len=L, with_v=with_v)
    A.seq_lens[2] = H - 5   # a short sequence (fast path) among them
    Bc = A.copy()
    Bc.pool_k = rng.integers(0, 256, A.pool_k.shape, dtype=np.uint8)
    if with_v:
        Bc.pool_v = rng.integers(0, 256, A.pool_v.shape, dtype=np.uint8)
    ga, gb, gc = GpuCase(A, dev), GpuCase(Bc, dev), GpuCase(Bc.copy(), dev)
    seq = torch.from_numpy(A.seq_lens).to(dev)
    req = torch.from_numpy(A.req_state).to(dev)
    topk = torch.zeros((B, K), dtype=torch.int32, device=dev)
    out_a = torch.zeros((B, K), dtype=torch.int32, device=dev)
    out_c = torch.zeros_like(out_a)
    miss = torch.zeros(B, dtype=torch.int32, device=dev)
    src = torch.zeros((B, K), dtype=torch.int64, device=dev)
    dst = torch.zeros((B, K), dtype=torch.int32, device=dev)

    def resolve(g, out, plan):
        kw = dict(miss_src=src, miss_dst=dst, miss_count=miss) if plan else {}
        return hs.make_swap_in_args(topk_ids=topk, seq_lens=seq, req_state=req,
                                    slot_tokens=g.tokens, slot_rows=g.rows, lru=g.lru,
                                    pool_rows=g.pool_rows, pool_k=g.pool_k, pool_v=g.pool_v,
                                    hot_k=g.hot_k, hot_v=g.hot_v, out_rows=out,
                                    overlap_prev=overlap and not plan, **kw)

    a_args, c_args = resolve(ga, out_a, True), resolve(gc, out_c, False)
    pools_b = [gb.pool_k, gb.pool_v] if with_v else [gb.pool_k]
    hots_b = [gb.hot_k, gb.hot_v] if with_v else [gb.hot_k]
    # pointer arrays are built outside graph capture (building them copies to the device)
    ptrs_b = (hs.layer_pointer_array(pools_b, dev), hs.layer_pointer_array(hots_b, dev))
    s = torch.cuda.Stream()

    def step():
        hs.swap_in_args(a_args, s)
        hs.gather_misses(pools_b, hots_b, src, dst, miss, has_v=with_v, stream=s, ptrs=ptrs_b,
                         overlap_prev=overlap)
        hs.swap_in_args(c_args, s)

    ts = synth.TopkStream(9, 0, B, K, L, 0.7)
    for n in range(6):
        topk.copy_(torch.from_numpy(ts.next()))
        torch.cuda.synchronize()
        if n < 3:
            with torch.cuda.stream(s):
                step()
        else:
            if n == 3:
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph, stream=s):
                    step()
                # capture does not run the work: replay once for this step
            graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out_a, out_c), n
        assert torch.equal(gb.hot_k, gc.hot_k), n
        if with_v:
            assert torch.equal(gb.hot_v, gc.hot_v), n
        assert torch.equal(ga.lru, gc.lru) and torch.equal(ga.tokens, gc.tokens), n


def test_empty_gather_launches_nothing(dev):
    hs = _hs()
    z64 = torch.zeros((0, 4), dtype=torch.int64, device=dev)
    z32 = torch.zeros((0, 4), dtype=torch.int32, device=dev)
    pool = torch.zeros((4, 16), dtype=torch.uint8, device=dev)
    hs.gather_misses([pool], [pool.clone()], z64, z32, torch.zeros(0, dtype=torch.int32, device=dev))
