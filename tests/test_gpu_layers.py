"""GPU parity for hs_swap_in_layers (every layer's swap-in in one launch, one
CTA per row and layer) and for hs_swap_in rows longer than 8192 slots, which
run on the same kernel: bit-exact against the CPU oracle run layer by layer
(outputs, miss counts, status bits, statistics, miss plans, slot tokens, LRU
order and hot-buffer bytes), through the C ABI."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import cases
import synth
from gpu_cases import GpuCase

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__

    __graft_entry__.build()
    return torch.device("cuda:0")


class Layers:
    """Several layers of one geometry, each with its own state and pool, stepped
    together through hs_swap_in_layers (or hs_swap_in per layer)."""

    def __init__(self, refs, dev, **gpu_kw):
        self.refs = refs
        self.gpus = [GpuCase(r.copy(), dev, **gpu_kw) for r in refs]
        self.dev = dev

    def args(self, ids, plan, overlap=False):
        import sparse_attention_kv_row_gb300 as hs

        dev = self.dev
        B, K = ids.shape[1:]
        res, layers = [], []
        for l, (g, ref) in enumerate(zip(self.gpus, self.refs)):
            o = dict(out=torch.full((B, K), 12345, dtype=torch.int32, device=dev),
                     miss=torch.full((B,), 777, dtype=torch.int32, device=dev),
                     status=torch.full((B,), 999, dtype=torch.int32, device=dev),
                     stats=torch.zeros(2, dtype=torch.int64, device=dev),
                     topk=torch.from_numpy(np.ascontiguousarray(ids[l])).to(dev))
            kw = {}
            if plan:
                o.update(miss_src=torch.full((B, K), cases.PLAN_FILL_SRC, dtype=torch.int64,
                                             device=dev),
                         miss_dst=torch.full((B, K), cases.PLAN_FILL_DST, dtype=torch.int32,
                                             device=dev),
                         miss_mask=torch.full((B, K), 7, dtype=torch.int32, device=dev))
                kw = {k: o[k] for k in ("miss_src", "miss_dst", "miss_mask")}
            num_real = (torch.tensor([ref.num_real], dtype=torch.int32, device=dev)
                        if ref.num_real >= 0 else None)
            o["num_real"] = num_real
            layers.append(hs.make_swap_in_args(
                topk_ids=o["topk"], seq_lens=torch.from_numpy(ref.seq_lens).to(dev, g.seq_dtype),
                req_state=torch.from_numpy(ref.req_state).to(dev, g.req_dtype),
                slot_tokens=g.tokens, slot_rows=g.rows, lru=g.lru, pool_rows=g.pool_rows,
                pool_k=g.pool_k, pool_v=g.pool_v, hot_k=g.hot_k, hot_v=g.hot_v,
                out_rows=o["out"], hot_size=ref.H, num_real=num_real, miss_count=o["miss"],
                stats=o["stats"], status=o["status"], max_seq_len=g._bound(),
                overlap_prev=overlap, **kw, **g.tables))
            res.append(o)
        return layers, res

    def step(self, ids, what="", plan=False, per_layer=False, overlap=False):
        import sparse_attention_kv_row_gb300 as hs

        layers, res = self.args(ids, plan, overlap)
        if per_layer:
            for a in layers:
                hs.swap_in_args(a)
        else:
            hs.swap_in_layers(layers)
        torch.cuda.synchronize()
        self.check(ids, res, what, plan)

    def check(self, ids, res, what, plan):
        names = ("out", "miss", "status", "stats", "miss_src", "miss_dst", "miss_mask")
        for l, (g, ref) in enumerate(zip(self.gpus, self.refs)):
            ref.topk = ids[l]
            r = cases.run_oracle(ref, plan=plan)
            o = res[l]
            got = [o["out"], o["miss"], o["status"], o["stats"]]
            if plan:
                got += [o["miss_src"], o["miss_dst"], o["miss_mask"]]
            for name, x, y in zip(names, got, r):
                x = x.cpu().numpy()
                if name == "stats":
                    x = x.astype(np.uint64)
                np.testing.assert_array_equal(x, y, err_msg=f"{name} layer {l} {what}")
            g.assert_matches(ref, f"layer {l} {what}")


def same_geometry_cases(rng, NL, **kw):
    seed = int(rng.integers(1 << 30))
    refs = []
    for l in range(NL):
        r = cases.random_case(np.random.default_rng(seed + l), **kw)
        refs.append(r)
    return refs


@pytest.mark.parametrize("seed", range(24))
def test_layers_random_tiny_with_corruption(dev, seed):
    rng = np.random.default_rng(9000 + seed)
    NL = int(rng.integers(1, 5))
    H = int(rng.integers(1, 40))
    K = int(rng.integers(1, H + 1))
    B = int(rng.integers(1, 6))
    S = int(rng.choice([1, 3, 4, 16, 17, 132, 656]))
    seq = rng.integers(1, 4 * H + 3, size=B)
    refs = same_geometry_cases(rng, NL, B=B, K=K, H=H, S=S, R=B + 2, seq_len=seq,
                               P=8 * H + 8, with_v=bool(seed % 3 == 0))
    nr = int(rng.choice([B, max(0, B - 1)])) if seed % 2 else -1
    for r in refs:   # num_real is given by every layer or by none
        r.num_real = nr
    ls = Layers(refs, dev, pool_in_host=bool(seed % 4 == 1),
                seq_dtype=torch.int32 if seed % 2 else torch.int64,
                req_dtype=torch.int32 if seed % 5 == 0 else torch.int64)
    prev = [None] * NL
    for step in range(5):
        ids = []
        for l in range(NL):
            ids.append(cases.random_ids(rng, refs[l], prev=prev[l]))
            prev[l] = ids[-1]
        ids = np.stack(ids)
        if step >= 3:
            for l in range(NL):
                cases.corrupt(np.random.default_rng(seed * 7 + step + 100 * l), refs[l])
                ls.gpus[l].push_state(refs[l])
        ls.step(ids, f"seed={seed} step={step}", plan=seed % 2 == 0)


@pytest.mark.parametrize("H,K,S,B,NL,with_v,host", [
    (1000, 700, 656, 5, 3, False, False),
    (2500, 2500, 132, 3, 2, False, True),     # K == H, 4-byte path, pinned host pools
    (4096, 2048, 656, 4, 2, True, False),     # K and V
    (3001, 1237, 17, 2, 3, False, False),     # byte path, odd sizes
    (777, 33, 2048, 3, 2, False, True),
])
def test_layers_multi_tile(dev, H, K, S, B, NL, with_v, host):
    rng = np.random.default_rng(H * 7 + K)
    L = 8 * H
    refs = same_geometry_cases(rng, NL, B=B, K=K, H=H, S=S, R=B + 1, seq_len=L,
                               with_v=with_v, width_pad=3)
    ls = Layers(refs, dev, pool_in_host=host)
    ts = [synth.TopkStream(H + l, 0, B, K, L, 0.6) for l in range(NL)]
    for step in range(4):
        ls.step(np.stack([t.next() for t in ts]), f"step {step}", plan=True)
    ls.step(np.stack([cases.random_ids(rng, r) for r in refs]), "mixed", plan=True)


@pytest.mark.parametrize("H,K,per_layer", [(16384, 300, True), (32767, 2048, True),
                                           (20000, 1500, False), (32767, 3000, True)])
def test_hot_sizes_above_8192(dev, H, K, per_layer):
    """hot_size 8193..32767: hs_swap_in sends such rows to the one-CTA kernel
    (slot tokens and rows read from global memory when they do not fit)."""
    rng = np.random.default_rng(H + K)
    B = 2
    L = 3 * H
    refs = same_geometry_cases(rng, 1 if per_layer else 2, B=B, K=K, H=H, S=16, R=B + 1,
                               seq_len=L)
    ls = Layers(refs, dev)
    ts = [synth.TopkStream(7 + l, 0, B, K, L, 0.5) for l in range(len(refs))]
    for step in range(3):
        ls.step(np.stack([t.next() for t in ts]), f"step {step}", plan=True,
                per_layer=per_layer)
    # corruption and mixed ids at the largest size
    for l, r in enumerate(refs):
        cases.corrupt(np.random.default_rng(3 + l), r)
        ls.gpus[l].push_state(r)
    ls.step(np.stack([cases.random_ids(rng, r) for r in refs]), "mixed", plan=True,
            per_layer=per_layer)


def test_layers_block_tables(dev):
    """Source and resident block tables, per layer, through the layers call."""
    rng = np.random.default_rng(44)
    NL, B, K, H, L, bs = 3, 3, 256, 700, 6000, 16
    refs = []
    for l in range(NL):
        r = cases.random_case(np.random.default_rng(50 + l), B=B, K=K, H=H, S=32, R=B + 1,
                              seq_len=L)
        R = r.lru.shape[0]
        nblk = (L + bs - 1) // bs
        P = r.pool_k.shape[0]
        src = np.random.default_rng(60 + l).integers(1, P // bs, size=(R, nblk)).astype(np.int32)
        src[:, 5] = 0   # unmapped blocks
        res = np.full((R, nblk), -1, np.int32)
        res[:, -3:] = np.arange(3, dtype=np.int32) + 2
        res[:, 7] = 0   # the null block
        r.tables = dict(src_block_table=src, src_block_size=bs, res_block_table=res,
                        res_block_size=bs, res_null_block=0)
        refs.append(r)
    ls = Layers(refs, dev)
    ts = [synth.TopkStream(70 + l, 0, B, K, L, 0.6) for l in range(NL)]
    for step in range(3):
        ls.step(np.stack([t.next() for t in ts]), f"step {step}", plan=True)
    ls.step(np.stack([cases.random_ids(rng, r) for r in refs]), "mixed", plan=True)


def test_layers_match_per_layer_calls_at_decode_shape(dev):
    """The decode shape (32 rows, top-k 2048, hot size 4096, 656 B rows) over
    three layers with early start: the layers call and three hs_swap_in calls
    give the oracle's results."""
    rng = np.random.default_rng(8)
    NL, B, K, H, L = 3, 32, 2048, 4096, 20000
    refs = same_geometry_cases(rng, NL, B=B, K=K, H=H, S=656, R=B, seq_len=L)
    ls = Layers(refs, dev)
    ts = [synth.TopkStream(90 + l, 0, B, K, L, 0.9) for l in range(NL)]
    for step in range(4):
        ls.step(np.stack([t.next() for t in ts]), f"step {step}", plan=step == 3,
                per_layer=step == 1, overlap=step >= 2)
        if step == 0:
            assert all(int(g.lru.shape[0]) == B for g in ls.gpus)


def test_layers_graph_capture(dev):
    """The layers call captured in a CUDA graph and replayed matches the oracle."""
    import sparse_attention_kv_row_gb300 as hs

    rng = np.random.default_rng(12)
    NL, B, K, H, L = 4, 3, 128, 512, 5000
    refs = same_geometry_cases(rng, NL, B=B, K=K, H=H, S=656, R=B, seq_len=L)
    ls = Layers(refs, dev)
    ts = [synth.TopkStream(30 + l, 0, B, K, L, 0.5) for l in range(NL)]
    ids = np.stack([t.next() for t in ts])
    layers, res = ls.args(ids, plan=False)
    arr = hs.layer_args_array(layers)
    s = torch.cuda.Stream()
    snap = [(g.tokens.clone(), g.lru.clone(), g.hot_k.clone()) for g in ls.gpus]
    with torch.cuda.stream(s):
        hs.swap_in_layers(arr, stream=s)   # one eager call first (kernel set-up)
    torch.cuda.synchronize()
    for g, (t, lr, hk) in zip(ls.gpus, snap):
        g.tokens.copy_(t); g.lru.copy_(lr); g.hot_k.copy_(hk)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        hs.swap_in_layers(arr, stream=s)
    torch.cuda.synchronize()
    for step in range(3):
        if step:
            ids = np.stack([t.next() for t in ts])
            for l in range(NL):
                res[l]["topk"].copy_(torch.from_numpy(ids[l]))
        for o in res:
            o["stats"].zero_()
        graph.replay()
        torch.cuda.synchronize()
        ls.check(ids, res, f"graph step {step}", plan=False)


@pytest.mark.parametrize("which,H", [(0, 600), (1, 600), (0, 12000), (1, 12000)])
def test_layers_forced_timeout(dev, which, H):
    """Every full-path row gives up one bounded wait at once (the copy is still
    waited out): the row reports exactly HS_ST_TIMEOUT, miss count 0, and
    nothing else is written; padding and short rows run as usual; a normal
    call afterwards matches the oracle.  H=12000 goes through hs_swap_in."""
    import oracle
    import sparse_attention_kv_row_gb300 as hs

    rng = np.random.default_rng(70 + which)
    NL, B, K, L = 2, 4, 200, 4 * H
    refs = same_geometry_cases(rng, NL, B=B, K=K, H=H, S=64, R=B + 1, seq_len=L)
    for r in refs:
        r.seq_lens[1] = H - 1   # short sequence
        r.req_state[2] = -1     # padding
    ls = Layers(refs, dev)
    ts = [synth.TopkStream(80 + l, 0, B, K, L, 0.5) for l in range(NL)]
    ls.step(np.stack([t.next() for t in ts]), "warm")
    ids = np.stack([t.next() for t in ts])
    before = [(g.tokens.clone(), g.lru.clone(), g.hot_k.clone()) for g in ls.gpus]
    layers, res = ls.args(ids, plan=True)
    if H > 8192:
        for a in layers:
            hs.swap_in_timeout_selftest(a, which=which)
    else:
        hs.swap_in_layers_timeout_selftest(layers, which=which)
    torch.cuda.synchronize()
    for l, (g, o) in enumerate(zip(ls.gpus, res)):
        assert torch.equal(g.tokens, before[l][0]) and torch.equal(g.lru, before[l][1])
        assert torch.equal(g.hot_k, before[l][2])
        assert int(o["stats"].abs().sum()) == 0
        st, ms, out = (o["status"].cpu().numpy(), o["miss"].cpu().numpy(),
                       o["out"].cpu().numpy())
        for b in (0, 3):
            assert st[b] == oracle.ST_TIMEOUT and ms[b] == 0 and np.all(out[b] == 12345)
            assert np.all(o["miss_mask"][b].cpu().numpy() == 7)
        probe = refs[l].copy()
        probe.topk = ids[l]
        r_out, r_miss, r_status, _ = cases.run_oracle(probe)
        for b in (1, 2):
            np.testing.assert_array_equal(out[b], r_out[b])
            assert ms[b] == r_miss[b] and st[b] == r_status[b]
    ls.step(ids, "after the forced time-out", plan=True)


def test_layers_argument_errors(dev):
    """Layers must agree in geometry; empty calls launch nothing."""
    import sparse_attention_kv_row_gb300 as hs

    rng = np.random.default_rng(5)
    refs = same_geometry_cases(rng, 2, B=2, K=8, H=16, S=16, R=3, seq_len=100)
    ls = Layers(refs, dev)
    ts = [synth.TopkStream(1 + l, 0, 2, 8, 100, 0.5) for l in range(2)]
    ids = np.stack([t.next() for t in ts])
    layers, _ = ls.args(ids, plan=False)
    layers[1].lru_stride += 1
    with pytest.raises(hs.HisparseError):
        hs.swap_in_layers(layers)
    layers, _ = ls.args(ids, plan=False)
    layers[1].stats = None
    with pytest.raises(hs.HisparseError):
        hs.swap_in_layers(layers)
    hs.swap_in_layers([])


def test_unsupported_sizes_are_refused(dev):
    """A row whose state cannot fit one CTA's shared memory is refused before
    any launch (HS_ERR_UNSUPPORTED), and hot_size above 32767 too."""
    import sparse_attention_kv_row_gb300 as hs

    assert hs.swap_in_smem_bytes(32767, 32767) > 227 * 1024
    assert hs.swap_in_smem_bytes(2048, 32767) <= 227 * 1024
    assert hs.swap_in_smem_bytes(10, 32768) == 0
    rng = np.random.default_rng(1)
    ref = cases.random_case(rng, B=1, K=20000, H=32767, S=16, R=1, seq_len=40000, P=40000)
    ls = Layers([ref], dev)
    layers, _ = ls.args(np.zeros((1, 1, 20000), np.int32), plan=False)
    with pytest.raises(hs.HisparseError) as e:
        hs.swap_in_args(layers[0])
    assert e.value.code == 2
