"""Mirror a numpy swap-in Case on the GPU and step it through the C ABI.

Test helper only: inputs come from tests/cases.py (seeded, host memory); the
GPU copy is stepped with sparse_attention_kv_row_gb300.swap_in and compared
with the oracle stepping the host copy.
"""
from __future__ import annotations

import numpy as np
import torch

import cases
import sparse_attention_kv_row_gb300 as hs


class GpuCase:
    def __init__(self, case: cases.Case, dev, *, pool_in_host=False, seq_dtype=torch.int64,
                 req_dtype=torch.int64, num_real_on_device=True, seq_bound="auto"):
        # seq_bound: the max_seq_len passed to the library; "auto" passes the case's
        # own bound, or its longest sequence when it has none (the compact hash)
        self.case = case
        self.dev = dev
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
        self.tokens = t(case.tokens)
        self.rows = t(case.rows)
        self.lru = t(case.lru)
        self.pool_rows = t(case.pool_rows)
        if pool_in_host:
            self.pool_k = torch.from_numpy(case.pool_k.copy()).pin_memory()
            self.pool_v = (torch.from_numpy(case.pool_v.copy()).pin_memory()
                           if case.pool_v is not None else None)
        else:
            self.pool_k = t(case.pool_k)
            self.pool_v = t(case.pool_v) if case.pool_v is not None else None
        self.hot_k = t(case.hot_k)
        self.hot_v = t(case.hot_v) if case.hot_v is not None else None
        self.seq_dtype, self.req_dtype = seq_dtype, req_dtype
        self.num_real_on_device = num_real_on_device
        self.seq_bound = seq_bound
        self.tables = {k: (t(v) if isinstance(v, np.ndarray) else v)
                       for k, v in case.tables.items()}

    def step(self, topk: np.ndarray, stream=None, plan=False):
        c = self.case
        B, K = topk.shape
        dev = self.dev
        out = torch.full((B, K), 12345, dtype=torch.int32, device=dev)
        miss = torch.full((B,), 777, dtype=torch.int32, device=dev)
        status = torch.full((B,), 999, dtype=torch.int32, device=dev)
        stats = torch.zeros(2, dtype=torch.int64, device=dev)
        kw = {}
        if plan:
            kw = dict(miss_src=torch.full((B, K), cases.PLAN_FILL_SRC, dtype=torch.int64, device=dev),
                      miss_dst=torch.full((B, K), cases.PLAN_FILL_DST, dtype=torch.int32, device=dev),
                      miss_mask=torch.full((B, K), 7, dtype=torch.int32, device=dev))
        num_real = None
        if c.num_real >= 0:
            num_real = torch.tensor([c.num_real], dtype=torch.int32, device=dev)
        hs.swap_in(topk_ids=torch.from_numpy(np.ascontiguousarray(topk)).to(dev),
                   seq_lens=torch.from_numpy(c.seq_lens).to(dev, self.seq_dtype),
                   req_state=torch.from_numpy(c.req_state).to(dev, self.req_dtype),
                   slot_tokens=self.tokens, slot_rows=self.rows, lru=self.lru,
                   pool_rows=self.pool_rows, pool_k=self.pool_k, pool_v=self.pool_v,
                   hot_k=self.hot_k, hot_v=self.hot_v, out_rows=out, hot_size=c.H,
                   num_real=num_real, miss_count=miss, stats=stats, status=status,
                   stream=stream, max_seq_len=self._bound(), **kw, **self.tables)
        torch.cuda.synchronize()
        res = (out.cpu().numpy(), miss.cpu().numpy(), status.cpu().numpy(),
               stats.cpu().numpy().astype(np.uint64))
        if plan:
            res += tuple(kw[k].cpu().numpy() for k in ("miss_src", "miss_dst", "miss_mask"))
        return res

    def _bound(self):
        if self.seq_bound != "auto":
            return int(self.seq_bound)
        return int(self.case.max_seq_len or max(1, int(np.max(self.case.seq_lens))))

    def assert_matches(self, ref: cases.Case, what=""):
        np.testing.assert_array_equal(self.tokens.cpu().numpy(), ref.tokens,
                                      err_msg=f"slot_tokens {what}")
        np.testing.assert_array_equal(self.lru.cpu().numpy(), ref.lru, err_msg=f"lru {what}")
        np.testing.assert_array_equal(self.hot_k.cpu().numpy(), ref.hot_k,
                                      err_msg=f"hot_k {what}")
        if self.hot_v is not None:
            np.testing.assert_array_equal(self.hot_v.cpu().numpy(), ref.hot_v,
                                          err_msg=f"hot_v {what}")

    def push_state(self, ref: cases.Case):
        """Overwrite device state with the host copy (after host-side corruption)."""
        self.tokens.copy_(torch.from_numpy(ref.tokens))
        self.rows.copy_(torch.from_numpy(ref.rows))
        self.lru.copy_(torch.from_numpy(ref.lru))
        self.pool_rows.copy_(torch.from_numpy(ref.pool_rows))


def step_both(g: GpuCase, ref: cases.Case, topk: np.ndarray, what="", plan=False):
    ref.topk = topk
    r = cases.run_oracle(ref, plan=plan)
    o = g.step(topk, plan=plan)
    names = ("out", "miss_count", "status", "stats", "miss_src", "miss_dst", "miss_mask")
    for name, x, y in zip(names, o, r):
        np.testing.assert_array_equal(x, y, err_msg=f"{name} {what}")
    g.assert_matches(ref, what)
    return o
