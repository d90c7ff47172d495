"""Seeded synthetic inputs for the HiSparse swap-in and the KV-row movers.

This module serves both the CUDA path's tests/benchmark and the CPU oracle.
It holds none of the method's arithmetic: only counter-based byte streams,
seeded top-k id sequences and the initial (cold) state layout.

Byte streams.  Byte ``j`` of row ``x`` in stream ``key`` is byte ``j % 4``
(little endian) of the 32-bit word ``fmix32(w XOR fmix32(key))`` with word
index ``w = x * ceil(S/4) + j // 4``.  ``fmix32`` is the 32-bit finaliser of
Austin Appleby's MurmurHash3 (public domain).  The numpy and torch versions
compute the same integers, so a pool generated on the GPU can be re-derived
row by row on the CPU.

Top-k sequences.  Per (seed, layer, row): step 0 draws K distinct ids uniformly
from [0, seq_len); step s+1 keeps exactly round(reuse*K) ids sampled without
replacement from step s, draws the rest uniformly from [0, seq_len) minus
step s's set, and shuffles the row.  The newest token (seq_len-1) appears only
when drawn.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

_M32 = 0xFFFFFFFF


# ---------------------------------------------------------------- byte streams
def fmix32_np(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, dtype=np.uint32).copy()
    x ^= x >> np.uint32(16)
    x *= np.uint32(0x85EBCA6B)
    x ^= x >> np.uint32(13)
    x *= np.uint32(0xC2B2AE35)
    x ^= x >> np.uint32(16)
    return x


def stream_key(*parts: int) -> int:
    """Fold integers into one 32-bit stream key."""
    k = np.uint32(0x243F6A88)
    for p in parts:
        k = fmix32_np(np.array([int(k) ^ (int(p) & _M32)], dtype=np.uint32))[0]
    return int(k)


def row_bytes_np(key: int, rows, row_bytes: int) -> np.ndarray:
    """uint8 [len(rows), row_bytes]: the stream's bytes for the given row ids."""
    rows = np.asarray(rows, dtype=np.int64).reshape(-1)
    W = (row_bytes + 3) // 4
    assert rows.size == 0 or (int(rows.max()) + 1) * W <= 1 << 32, "word index exceeds 32 bits"
    w = (rows[:, None] * W + np.arange(W, dtype=np.int64)[None, :]).astype(np.uint32)
    kk = fmix32_np(np.array([key], dtype=np.uint32))[0]
    words = fmix32_np(w ^ kk)
    return words.view(np.uint8).reshape(rows.size, W * 4)[:, :row_bytes].copy()


def _mul32_t(x, c: int):
    # (x * c) mod 2^32 for int64 tensors holding values in [0, 2^32), without
    # overflowing int64: split c into 16-bit halves.
    lo = x * (c & 0xFFFF)
    hi = ((x * (c >> 16)) & 0xFFFF) << 16
    return (lo + hi) & _M32


def fmix32_torch(x):
    x = x ^ (x >> 16)
    x = _mul32_t(x, 0x85EBCA6B)
    x = x ^ (x >> 13)
    x = _mul32_t(x, 0xC2B2AE35)
    return x ^ (x >> 16)


def fill_rows_torch(dst, key: int, first_row: int = 0, chunk_words: int = 1 << 26):
    """Fill a uint8 tensor ``dst`` [n, S] (any device, rows contiguous, S % 4 == 0)
    with the stream's bytes of rows first_row .. first_row+n-1."""
    import torch

    n, S = dst.shape
    assert S % 4 == 0 and dst.is_contiguous()
    W = S // 4
    assert (first_row + n) * W <= 1 << 32, "word index exceeds 32 bits"
    flat = dst.view(torch.int32).view(-1)
    kk = int(fmix32_np(np.array([key], dtype=np.uint32))[0])
    base = first_row * W
    total = n * W
    for s in range(0, total, chunk_words):
        e = min(total, s + chunk_words)
        w = torch.arange(base + s, base + e, dtype=torch.int64, device=dst.device)
        v = fmix32_torch(w ^ kk)
        v = v - (v >= (1 << 31)).to(torch.int64) * (1 << 32)  # to signed 32-bit pattern
        flat[s:e] = v.to(torch.int32)
    return dst


# ------------------------------------------------------------ top-k sequences
def _draw_fresh(rng, n: int, seq_len: int, exclude: np.ndarray) -> np.ndarray:
    got = np.empty(0, dtype=np.int64)
    while got.size < n:
        cand = rng.integers(0, seq_len, size=2 * (n - got.size) + 8)
        cand = cand[~np.isin(cand, exclude)]
        cand = cand[~np.isin(cand, got)]
        _, first = np.unique(cand, return_index=True)
        cand = cand[np.sort(first)]
        got = np.concatenate([got, cand[: n - got.size]])
    return got


class TopkStream:
    """Seeded per-row top-k id sequence (see module docstring)."""

    def __init__(self, seed: int, layer: int, batch: int, top_k: int, seq_len,
                 reuse: float):
        self.batch, self.top_k, self.reuse = batch, top_k, reuse
        self.seq_len = np.broadcast_to(np.asarray(seq_len, dtype=np.int64), (batch,)).copy()
        assert np.all(self.seq_len >= top_k), "need seq_len >= top_k for distinct ids"
        self.rngs = [np.random.default_rng([seed, layer, b]) for b in range(batch)]
        self.prev = [None] * batch

    def next(self) -> np.ndarray:
        K = self.top_k
        out = np.empty((self.batch, K), dtype=np.int32)
        for b in range(self.batch):
            rng, L = self.rngs[b], int(self.seq_len[b])
            if self.prev[b] is None:
                ids = _draw_fresh(rng, K, L, np.empty(0, dtype=np.int64))
            else:
                keep_n = int(round(self.reuse * K))
                keep = rng.choice(self.prev[b], size=keep_n, replace=False)
                fresh = _draw_fresh(rng, K - keep_n, L, self.prev[b])
                ids = np.concatenate([keep, fresh])
            ids = rng.permutation(ids)
            self.prev[b] = ids.astype(np.int64)
            out[b] = ids
        return out


# ------------------------------------------------------------------ state
def cold_state(num_states: int, hot_size: int, width: int | None = None, seed: int | None = None):
    """Cold start: lru[r] = [0..H), slot_tokens = -1, slot_rows[r][s] = r*(H+1)+s,
    or a seeded permutation of those hot rows when ``seed`` is given.
    Returns (slot_tokens int32 [R,W], slot_rows int32 [R,W], lru int16 [R,H])."""
    H = hot_size
    W = width if width is not None else H + 1
    assert W >= H + 1
    tokens = np.full((num_states, W), -1, dtype=np.int32)
    rows = np.full((num_states, W), -1, dtype=np.int32)
    base = np.arange(num_states * (H + 1), dtype=np.int64).reshape(num_states, H + 1)
    if seed is not None:
        base = np.random.default_rng(seed).permutation(base.reshape(-1)).reshape(base.shape)
    rows[:, : H + 1] = base.astype(np.int32)
    lru = np.tile(np.arange(H, dtype=np.int16), (num_states, 1))
    return tokens, rows, lru


# ------------------------------------------------------------------ configs
@dataclasses.dataclass(frozen=True)
class SwapInConfig:
    name: str
    batch: int
    top_k: int
    hot_size: int
    row_bytes: int
    seq_len: int
    reuse: float
    layers: int
    pool_in_host: bool
    seed: int

    @property
    def pool_rows_per_state(self) -> int:
        return self.seq_len

    @property
    def warm_steps(self) -> int:
        fresh = max(1, self.top_k - int(round(self.reuse * self.top_k)))
        return math.ceil(self.hot_size / fresh) + 1


# The five workloads (sizes as stated for the benchmark configurations).
TINY = SwapInConfig("tiny swap-in B=2 K=16 H=64 S=656 HBM pool 1024 rows", 2, 16, 64, 656,
                    1024, 0.5, 1, False, 101)
DSV32 = SwapInConfig("DeepSeek-V3.2-shaped swap-in B=32 K=2048 H=4096 S=656 HBM pool 32x128K, "
                     "61 layers, 90% reuse", 32, 2048, 4096, 656, 131072, 0.9, 61, False, 303)
INDEXER = SwapInConfig("indexer-row swap-in B=64 K=2048 H=2048 S=132 pinned-host pool 64x64K, "
                       "80% reuse", 64, 2048, 2048, 132, 65536, 0.8, 1, True, 404)
STRESS = SwapInConfig("high-miss stress swap-in B=128 K=2048 H=2048 S=656 pinned-host pool "
                      "128x128K, 70% reuse", 128, 2048, 2048, 656, 131072, 0.7, 1, True, 505)
STORE_KV = dict(name="store_kv scatter: 4096 tokens, K and V [8 x 128] bf16 (2048 B rows) into "
                "two 2^20-row pools", n_tokens=4096, heads=8, head_dim=128, pool_rows=1 << 20,
                seed=202)
TRANSFER = dict(name="all-layer transfer_kv: 61 layers x 78,592 pairs of 656 B rows, pinned "
                "host -> HBM", layers=61, row_bytes=656, seed=606)


class TopkStreamTorch:
    """The same recipe as TopkStream, drawn with torch on any device (used for
    the large benchmark workloads): per row, step s+1 keeps exactly
    round(reuse*K) ids of step s chosen uniformly without replacement, draws the
    other ids uniformly without replacement from [0, seq_len) minus step s's
    set, and shuffles.  Rows are independent; ``rows`` may span many layers."""

    def __init__(self, seed: int, rows: int, top_k: int, seq_len: int, reuse: float, device):
        import torch

        assert seq_len >= 2 * top_k, "needs seq_len >= 2*top_k"
        self.rows, self.top_k, self.seq_len, self.reuse = rows, top_k, seq_len, reuse
        self.device = torch.device(device)
        self.gen = torch.Generator(device=self.device)
        self.gen.manual_seed(seed)
        self.prev = None

    def _distinct(self, n: int, N: int):
        """[rows, n] distinct uniform values from [0, N), each row independently."""
        import torch

        R, dev, g = self.rows, self.device, self.gen
        if n * n > N:  # dense: random keys, take the n smallest
            out = torch.empty((R, n), dtype=torch.int64, device=dev)
            for r0 in range(0, R, 64):
                r1 = min(R, r0 + 64)
                keys = torch.rand((r1 - r0, N), generator=g, device=dev)
                out[r0:r1] = keys.topk(n, dim=1, largest=False).indices
            return out
        # sparse: draw with replacement and redraw rows holding a repeat; with
        # n*n <= N a row is repeat-free with probability >= exp(-1/2)
        out = torch.randint(0, N, (R, n), generator=g, device=dev)
        while True:
            srt = out.sort(dim=1).values
            bad = (srt[:, 1:] == srt[:, :-1]).any(dim=1)
            nbad = int(bad.sum())
            if nbad == 0:
                return out
            out[bad] = torch.randint(0, N, (nbad, n), generator=g, device=dev)

    def next(self):
        import torch

        R, K, L, dev, g = self.rows, self.top_k, self.seq_len, self.device, self.gen
        if self.prev is None:
            ids = self._distinct(K, L)
        else:
            keep_n = int(round(self.reuse * K))
            order = torch.rand((R, K), generator=g, device=dev).argsort(dim=1)[:, :keep_n]
            kept = self.prev.gather(1, order)
            # the v-th element of [0, L) minus the sorted excluded set e is
            # v + #{j : e[j] - j <= v}
            e = self.prev.sort(dim=1).values
            shifted = e - torch.arange(K, device=dev)[None, :]
            v = self._distinct(K - keep_n, L - K)
            fresh = v + torch.searchsorted(shifted, v, right=True)
            ids = torch.cat([kept, fresh], dim=1)
        perm = torch.rand((R, K), generator=g, device=dev).argsort(dim=1)
        ids = ids.gather(1, perm)
        self.prev = ids
        return ids.to(torch.int32)
