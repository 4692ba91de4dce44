"""Host-side input generators (no attention arithmetic): the sparse top-k
lists hold what their docstring promises.  CPU only."""
import torch

from paged_varlen_flash_gb300 import workloads as W


def _rows(w):
    out = []
    for s, (sq, sk) in enumerate(zip(w.seqlens_q, w.seqlens_k)):
        for i in range(sq):
            out.append((sq, sk, i, sk - sq))
    return out


def test_topk_lists_are_distinct_visible_keys_without_junk():
    sq, sk = [1, 3, 2], [50, 400, 9]
    idx, lens = W.topk_lists(sq, sk, 64, seed=3)
    assert idx.dtype == torch.int32 and idx.shape == (sum(sq), 64)
    t = 0
    for q, k in zip(sq, sk):
        ctx = k - q
        for i in range(q):
            n = int(lens[t])
            assert n == min(64, i + ctx + 1)           # full lists when not ragged
            row = idx[t, :n]
            assert len(set(row.tolist())) == n         # distinct
            assert int(row.min()) >= 0 and int(row.max()) <= i + ctx
            assert torch.all(idx[t, n:] == -1)         # unused slots
            t += 1


def test_topk_lists_ragged_and_junk_entries_are_not_keys_of_the_row():
    sq, sk = [2, 4, 1], [300, 700, 40]
    idx, lens = W.topk_lists(sq, sk, 128, seed=5, ragged=True, junk=0.5)
    t, junk = 0, 0
    for q, k in zip(sq, sk):
        ctx = k - q
        for i in range(q):
            n = int(lens[t])
            assert 0 <= n <= 128
            row = idx[t, :n].tolist()
            keys = [j for j in row if 0 <= j <= i + ctx]
            junk += n - len(keys)
            for j in row:
                assert j == -1 or j >= 0
                if not (0 <= j <= i + ctx):
                    assert j == -1 or j >= i + ctx + 1   # -1, hidden, or past S_k
            t += 1
    assert junk > 0


def test_decode_topk_workload_shape_and_counts():
    w = W.make("decode_topk", values=False)
    assert w.topk_idx.shape == (256, 2048) and int(w.topk_len.min()) == 2048
    assert w.visible_pairs() == 256 * 2048
    assert w.kv_bytes_read() == 256 * 2048 * 1 * 128 * 2 * 2


def test_kv_keys_read_is_the_union_of_the_rows_visible_keys():
    # Brute force: mark every key some row of the sequence can see (causal,
    # window W keeps [i + ctx - W + 1, i + ctx]) and count the marks.
    for window in (0, 1, 7, 100, 5000):
        w = W.random_small(71 + window, num_seqs=5, sq=(1, 60), ctx=(0, 300), window=window,
                           poison=False)
        want = 0
        for sq, sk in zip(w.seqlens_q, w.seqlens_k):
            ctx = sk - sq
            seen = set()
            for i in range(sq):
                lo = max(0, i + ctx - window + 1) if window else 0
                seen.update(range(lo, i + ctx + 1))
            want += len(seen)
        assert w.kv_keys_read() == want, window
        assert w.kv_bytes_read() == want * w.hk * w.d * 2 * 2


def test_chunked_workload_reads_only_its_windows():
    w = W.make("chunked", values=False)
    full = sum(w.seqlens_k) * w.hk * w.d * 2 * 2
    assert 70e6 <= w.kv_bytes_read() <= 76e6 < full
