"""The benchmark's FLOP accounting: the number of visible (query, key) pairs
per head that the effective-TFLOP/s metric counts (4 * head_dim * n_q_heads
flops per pair: QK^T and PV, masked pairs excluded).

Pinned against a brute-force count of the bottom-right causal rule (query
row i of a chunk with prefix P sees keys j with j <= P + i, and with a window
W also j > P + i - W), and against the pair counts of two configurations
that follow from it in closed form: the tiny case (prefixes 0 and 37, chunks
5 and 40: 15 + 2300 = 2315 pairs) and the mixed batch's prompt rows (one
4097-token prompt as chunks 2048 / 2048 / 1: 2,098,176 + 6,292,480 + 4097 =
8,394,753 pairs).
"""
import numpy as np
import pytest

import bench
import workloads as W


def brute_pairs(prefix_lens, chunk_lens, window):
    n = 0
    for P, c in zip(prefix_lens, chunk_lens):
        for i in range(c):
            p = P + i
            for j in range(p + 1):
                if window <= 0 or j > p - window:
                    n += 1
    return n


def test_tiny_case_pairs():
    assert bench.visible_pairs([0, 37], [5, 40], 0) == 2315


def test_mixed_prompt_rows_pairs():
    assert bench.visible_pairs([0, 2048, 4096], [2048, 2048, 1], 0) == 8_394_753


@pytest.mark.parametrize("window", [0, 1, 7, 64])
def test_visible_pairs_matches_brute_force(window):
    rng = np.random.default_rng(window)
    P = rng.integers(0, 150, size=9).tolist()
    C = rng.integers(0, 40, size=9).tolist()
    assert bench.visible_pairs(P, C, window) == brute_pairs(P, C, window)


def test_row_samples_sum_to_the_whole():
    b = W.make_batch([0, 37, 300, 5], [5, 40, 1, 64], 4, 2, 64, 16, seed=7, window=100)
    tok = np.arange(b.total_q)
    assert bench.rows_pairs(b, tok, np.zeros_like(tok)) == \
        bench.visible_pairs(b.prefix_lens, b.chunk_lens, b.window)


def test_split_work_divides_the_mixed_batch():
    """The mixed batch's 2048-token chunks go to the tensor cores (2,098,176 +
    6,292,480 pairs); its 1-token chunk and the 31 decode rows (chunk_len * G
    = 4 <= 16 rows) go to the row kernel, which reads every visible key's K
    and V once per KV head."""
    b = W.mixed_batch()
    tc_pairs, row_bytes = bench.split_work(b)
    assert tc_pairs == 2_098_176 + 6_292_480
    c = b.chunk_lens
    rows = c == 1
    L = (b.prefix_lens + c)[rows].astype(np.int64)
    D, Hkv, Hq = b.head_dim, b.n_kv_heads, b.n_q_heads
    pages = sum(-(-int(l) // b.page_size) for l in L)
    expect = int(L.sum()) * Hkv * D * 4 + int(rows.sum()) * Hq * (4 * D + 4) + 4 * pages
    assert row_bytes == expect


@pytest.mark.parametrize("window", [0, 5, 300])
def test_split_work_matches_brute_force(window):
    """Tensor-core pairs by brute force over the chunks longer than the row
    path takes; row bytes from each row's visible keys counted one by one."""
    b = W.make_batch([0, 37, 300, 5, 900, 17], [5, 40, 1, 64, 2, 3], 8, 2, 64, 16, seed=7,
                     window=window)
    rmax = bench.row_max_chunk(b)
    assert rmax == 4
    c, P = b.chunk_lens, b.prefix_lens
    tc = c > rmax
    tc_pairs, row_bytes = bench.split_work(b)
    assert tc_pairs == brute_pairs(P[tc], c[tc], window)
    keys = 0
    for Pb, cb in zip(P[~tc], c[~tc]):
        first = max(0, Pb - window + 1) if window > 0 else 0
        keys += len(range(first, Pb + cb))
    pages = sum(-(-int(Pb + cb) // 16) for Pb, cb in zip(P[~tc], c[~tc]))
    n_rows = int(c[~tc].sum())
    assert row_bytes == keys * 2 * 64 * 4 + n_rows * 8 * (4 * 64 + 4) + 4 * pages


def test_launches_per_step():
    """Library kernels per step (one call with the new K/V rows): the GQA
    step launches the planner with the append beside it and the tensor-core
    kernel; a decode-only step of 31 sequences the append, the row kernel
    (which plans itself) and the combine; the mixed step four, or two when
    its decode rows joined the tensor cores."""
    assert bench.launches_per_step(W.gqa_prefill()) == 2
    assert bench.launches_per_step(W.decode_rows()) == 3
    assert bench.launches_per_step(W.mixed_batch()) == 4
    assert bench.launches_per_step(W.mixed_batch(), rows_on_tensor_cores=True) == 2
    # more than 512 decode-only sequences: the planner (with the append
    # beside it), the row kernel and the combine
    b = W.make_batch([100] * 513, [1] * 513, 4, 4, 64, 16, seed=3)
    assert bench.launches_per_step(b) == 3
