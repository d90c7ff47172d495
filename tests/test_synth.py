"""The seeded input generators: reproducible, and identical between the numpy
and torch implementations (so GPU-generated pools can be re-derived on CPU)."""
import numpy as np
import torch

import synth


def test_fmix32_known_values():
    # MurmurHash3 fmix32 of 0 is 0; of 1 is 0x514E28B7 (finaliser applied to 1).
    assert int(synth.fmix32_np(np.array([0], np.uint32))[0]) == 0
    assert int(synth.fmix32_np(np.array([1], np.uint32))[0]) == 0x514E28B7


def test_torch_matches_numpy_bytes():
    key = synth.stream_key(3, 7)
    for S in (4, 132, 656):
        rows = np.arange(17, 40)
        ref = synth.row_bytes_np(key, rows, S)
        t = torch.empty((rows.size, S), dtype=torch.uint8)
        synth.fill_rows_torch(t, key, first_row=17, chunk_words=97)
        np.testing.assert_array_equal(t.numpy(), ref)


def test_row_bytes_odd_size_is_prefix():
    key = synth.stream_key(1)
    a = synth.row_bytes_np(key, [5], 7)
    b = synth.row_bytes_np(key, [5], 8)
    np.testing.assert_array_equal(a[0], b[0, :7])


def test_topk_stream_reuse_and_distinct():
    ts = synth.TopkStream(5, 2, 3, 64, 1000, 0.75)
    prev = ts.next()
    for _ in range(5):
        cur = ts.next()
        for b in range(3):
            assert len(set(cur[b].tolist())) == 64
            assert np.all((cur[b] >= 0) & (cur[b] < 1000))
            assert len(set(cur[b].tolist()) & set(prev[b].tolist())) == 48
        prev = cur
    again = synth.TopkStream(5, 2, 3, 64, 1000, 0.75).next()
    first = synth.TopkStream(5, 2, 3, 64, 1000, 0.75).next()
    np.testing.assert_array_equal(again, first)


def test_cold_state_layout():
    tok, rows, lru = synth.cold_state(3, 5)
    assert tok.shape == (3, 6) and np.all(tok == -1)
    assert rows[1].tolist() == list(range(6, 12))
    assert lru[2].tolist() == list(range(5))
    _, prow, _ = synth.cold_state(3, 5, seed=1)
    assert sorted(prow.reshape(-1).tolist()) == list(range(18))


def test_topk_stream_torch_recipe():
    ts = synth.TopkStreamTorch(3, 5, 64, 700, 0.75, "cpu")
    prev = ts.next().numpy()
    for _ in range(6):
        cur = ts.next().numpy()
        for b in range(5):
            s = set(cur[b].tolist())
            assert len(s) == 64 and min(s) >= 0 and max(s) < 700
            assert len(s & set(prev[b].tolist())) == 48
        prev = cur
    a = synth.TopkStreamTorch(3, 5, 64, 700, 0.75, "cpu")
    b = synth.TopkStreamTorch(3, 5, 64, 700, 0.75, "cpu")
    for _ in range(3):
        np.testing.assert_array_equal(a.next().numpy(), b.next().numpy())


def test_topk_stream_torch_fresh_is_uniform_over_complement():
    # the complement mapping covers every non-excluded id and never an excluded one
    ts = synth.TopkStreamTorch(4, 200, 8, 20, 0.5, "cpu")
    first = ts.next()
    second = ts.next().numpy()
    prev = first.numpy()
    seen = set()
    for r in range(200):
        fresh = set(second[r].tolist()) - set(prev[r].tolist())
        assert len(fresh) == 4
        seen |= fresh
    assert seen == set(range(20))
