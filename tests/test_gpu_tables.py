"""GPU parity for the block-table translation, the resident-block lookup and
the invalidation of rewritten tokens, against the CPU oracle element by element
(outputs, counters, status bits, miss plan, slot tokens, LRU order, hot bytes):
source tables with unmapped blocks, resident tables with a null block, both
together, repeated ids, short sequences, padding rows, a multi-tile size, and
invalidation with out-of-range state rows."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import cases
import oracle
from gpu_cases import GpuCase, step_both
from test_oracle_tables import block_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__

    __graft_entry__.build()
    return torch.device("cuda:0")


def _resident(rng, c, rbs=8, frac=0.3, null=5):
    R, L = c.pool_rows.shape
    nb = -(-L // rbs)
    res = np.full((R, nb), -1, np.int32)
    pick = rng.random((R, nb)) < frac
    res[pick] = rng.permutation(4000)[: pick.sum()] + 10
    res[0, 0] = null
    c.tables.update(res_block_table=res, res_block_size=rbs, res_null_block=null)


@pytest.mark.parametrize("kind", ["source", "source_unmapped", "resident", "both"])
def test_tables_parity(dev, kind):
    rng = np.random.default_rng(hash(kind) % 1000)
    ref = block_case(rng, B=4, K=60, H=150, L=900, bs=4,
                     unmapped=0.15 if kind in ("source_unmapped", "both") else 0.0)
    if kind == "resident":
        ref.tables = {}
        ref.pool_rows = np.stack([rng.permutation(ref.pool_k.shape[0])[:900]
                                  for _ in range(ref.pool_rows.shape[0])]).astype(np.int64)
    if kind in ("resident", "both"):
        _resident(rng, ref)
    ref.seq_lens[1] = 120          # a short sequence: fast path
    ref.num_real = 3               # the last row is padding
    g = GpuCase(ref.copy(), dev)
    prev = None
    for step in range(6):
        ids = cases.random_ids(rng, ref, prev=prev)
        prev = ids
        step_both(g, ref, ids, f"{kind} step {step}", plan=True)


def test_tables_multi_tile(dev):
    rng = np.random.default_rng(77)
    ref = block_case(rng, B=3, K=1500, H=3000, L=30000, bs=16, unmapped=0.05)
    _resident(rng, ref, rbs=64, frac=0.1)
    g = GpuCase(ref.copy(), dev)
    import synth
    ts = synth.TopkStream(4, 0, ref.B, ref.K, 30000, 0.8)
    for step in range(4):
        step_both(g, ref, ts.next(), f"step {step}", plan=True)


@pytest.mark.parametrize("H", [700, 2500])  # one chunk of 1024 slots; three with a ragged tail
def test_invalidate_parity(dev, H):
    import sparse_attention_kv_row_gb300 as hs

    rng = np.random.default_rng(8 + H)
    R = 9
    tok = rng.integers(-1, 500, (R, H + 4)).astype(np.int32)
    rows = rng.integers(-1, R + 2, 300).astype(np.int64)
    toks = rng.integers(-3, 500, 300).astype(np.int32)
    ref = tok.copy()
    st_ref = np.zeros(1, np.int32)
    oracle.invalidate_tokens(slot_tokens=ref, hot_size=H, state_rows=rows, tokens=toks,
                             status=st_ref)
    g = torch.from_numpy(tok).to(dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    hs.invalidate_tokens(g, torch.from_numpy(rows).to(dev), torch.from_numpy(toks).to(dev),
                         hot_size=H, status=st)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(g.cpu().numpy(), ref)
    assert st.item() == st_ref[0] == oracle.ST_BAD_INDEX
