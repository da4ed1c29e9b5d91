"""Pins for the oracle's non-causal and boolean-mask attention.

The AstrAI paged prefill entry point takes ``is_causal`` and an optional
boolean ``mask`` (True = keep) of shape [batch, 1, q_len, kv_len] (or
[batch, kv_len] on the decode path), indexed by the request-local query row
and key; its prefill-with-mask regression test runs a 4-D causal-pattern mask
with causality off.  Each check below ties the oracle to something other than
itself:

* a closed form: with Q = 0 every visible key gets the same weight, so with
  V_j = j the output is the mean of the visible key positions and lse is the
  log of their count; the visible sets are listed here with plain Python
  loops straight from the mask entries;
* equivalences: an explicit bottom-right causal mask with causality off equals
  the causal flag; an all-True mask equals no mask; a head-broadcast mask
  equals the same mask written out per head;
* brute force: a dense numpy softmax over all keys, masked with -inf,
  gathered by page-list expansion;
* argument rules: a window needs causal attention; keys past the mask's kv
  extent read as masked.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from test_oracle_pins import expand_slots


def position_batch(P, C, Hq, Hkv, D, ps, seed, window=0):
    """A batch whose queries are 0 and whose value rows hold their key
    position j in every lane (exact in bf16 for j <= 256)."""
    b = W.make_batch(P, C, Hq, Hkv, D, ps, seed=seed, window=window)
    b.q[:] = 0
    for s in range(b.batch):
        L = int(b.kv_lens[s])
        slots = expand_slots(b.kv_indptr, b.kv_indices, s, ps, L)
        Pb = int(b.prefix_lens[s])
        b.v_pool[slots[:Pb]] = W.bf16_bits(
            np.broadcast_to(np.arange(Pb, dtype=np.float32)[:, None, None], (Pb, Hkv, D)))
        t0 = int(b.qo_indptr[s])
        c = int(b.chunk_lens[s])
        b.v_new[t0:t0 + c] = W.bf16_bits(
            np.broadcast_to(np.arange(Pb, Pb + c, dtype=np.float32)[:, None, None],
                            (c, Hkv, D)))
    return b


def mask_entry(mask, b, h, i, j):
    """mask[b, h, i, j] with broadcasting over size-1 head / row dimensions."""
    if mask.ndim == 2:
        return j < mask.shape[1] and bool(mask[b, j])
    hh = 0 if mask.shape[1] == 1 else h
    if mask.shape[2] != 1 and i >= mask.shape[2]:
        return False
    ii = 0 if mask.shape[2] == 1 else i
    return j < mask.shape[3] and bool(mask[b, hh, ii, j])


def visible_keys(batch, b, i, h, causal, mask):
    P = int(batch.prefix_lens[b])
    L = int(batch.kv_lens[b])
    p = P + i
    keys = []
    for j in range(L):
        if causal and (j > p or (batch.window > 0 and j <= p - batch.window)):
            continue
        if mask is not None and not mask_entry(mask, b, h, i, j):
            continue
        keys.append(j)
    return keys


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("kind", [None, "2d", "4d_bcast", "4d_heads", "4d_q1"])
def test_mask_position_mean_closed_form(causal, kind):
    batch = position_batch([0, 37, 100, 5], [40, 1, 70, 0], 4, 2, 16, 16, seed=61)
    mask = None if kind is None else W.random_mask(batch, kind, seed=62, keep=0.5)
    _, _, _, out, lse = oracle.run_batch(batch, causal=causal, mask=mask)
    n_empty = 0
    for b in range(batch.batch):
        t0 = int(batch.qo_indptr[b])
        for i in range(int(batch.chunk_lens[b])):
            for h in range(batch.n_q_heads):
                keys = visible_keys(batch, b, i, h, causal, mask)
                if not keys:
                    n_empty += 1
                    assert (out[t0 + i, h] == 0).all() and lse[t0 + i, h] == -np.inf
                    continue
                np.testing.assert_allclose(out[t0 + i, h], np.mean(keys), rtol=0, atol=1e-9)
                np.testing.assert_allclose(lse[t0 + i, h], np.log(len(keys)), rtol=0,
                                           atol=1e-12)
    if kind is None:
        assert n_empty == 0


def test_windowed_causal_with_mask_closed_form():
    batch = position_batch([50, 0], [30, 64], 4, 1, 16, 8, seed=63, window=20)
    mask = W.random_mask(batch, "4d_heads", seed=64, keep=0.7)
    _, _, _, out, lse = oracle.run_batch(batch, mask=mask)
    for b in range(batch.batch):
        t0 = int(batch.qo_indptr[b])
        for i in range(int(batch.chunk_lens[b])):
            for h in range(batch.n_q_heads):
                keys = visible_keys(batch, b, i, h, True, mask)
                if keys:
                    np.testing.assert_allclose(out[t0 + i, h], np.mean(keys), atol=1e-9)
                    np.testing.assert_allclose(lse[t0 + i, h], np.log(len(keys)), atol=1e-12)
                else:
                    assert lse[t0 + i, h] == -np.inf


def test_explicit_causal_mask_equals_causal_flag():
    """The AstrAI regression shape: a 4-D bottom-right causal pattern given as
    a mask with causality off."""
    batch = W.make_batch([0, 300, 17], [96, 41, 128], 8, 2, 64, 16, seed=65)
    kv = int(-(-int(batch.kv_lens.max()) // 16) * 16)
    qmax = int(batch.chunk_lens.max())
    mask = np.zeros((batch.batch, 1, qmax, kv), bool)
    for b in range(batch.batch):
        P = int(batch.prefix_lens[b])
        for i in range(int(batch.chunk_lens[b])):
            mask[b, 0, i, :P + i + 1] = True
    _, _, _, o1, l1 = oracle.run_batch(batch, causal=False, mask=mask)
    _, _, _, o2, l2 = oracle.run_batch(batch)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


@pytest.mark.parametrize("causal", [True, False])
def test_all_true_mask_equals_no_mask(causal):
    batch = W.make_batch([10, 0], [20, 33], 4, 2, 64, 4, seed=66)
    for kind in ("2d", "4d_heads"):
        mask = np.ones_like(W.random_mask(batch, kind, seed=0))
        _, _, _, o1, l1 = oracle.run_batch(batch, causal=causal, mask=mask)
        _, _, _, o2, l2 = oracle.run_batch(batch, causal=causal)
        np.testing.assert_array_equal(o1, o2)
        np.testing.assert_array_equal(l1, l2)


def test_head_broadcast_equals_per_head_copy():
    batch = W.make_batch([64, 3], [30, 18], 8, 2, 64, 16, seed=67)
    m1 = W.random_mask(batch, "4d_bcast", seed=68)
    m2 = np.repeat(m1, batch.n_q_heads, axis=1)
    _, _, _, o1, l1 = oracle.run_batch(batch, mask=m1)
    _, _, _, o2, l2 = oracle.run_batch(batch, mask=m2)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def dense_masked(batch, k_pool, v_pool, causal, mask):
    """Dense softmax over all keys of each sequence, masked entries -inf."""
    Hq, Hkv, D = batch.n_q_heads, batch.n_kv_heads, batch.head_dim
    G = Hq // Hkv
    scale = batch.sm_scale if batch.sm_scale > 0 else 1.0 / np.sqrt(D)
    out = np.zeros((batch.total_q, Hq, D))
    lse = np.full((batch.total_q, Hq), -np.inf)
    for b in range(batch.batch):
        P, c = int(batch.prefix_lens[b]), int(batch.chunk_lens[b])
        L = P + c
        if c == 0:
            continue
        s = expand_slots(batch.kv_indptr, batch.kv_indices, b, batch.page_size, L)
        K = W.bf16_to_f32(k_pool[s]).astype(np.float64)
        V = W.bf16_to_f32(v_pool[s]).astype(np.float64)
        t0 = int(batch.qo_indptr[b])
        Q = W.bf16_to_f32(batch.q[t0:t0 + c]).astype(np.float64)
        for h in range(Hq):
            keep = np.ones((c, L), bool)
            if causal:
                keep &= np.arange(L)[None, :] <= (P + np.arange(c))[:, None]
            if mask is not None:
                for i in range(c):
                    keep[i] &= [mask_entry(mask, b, h, i, j) for j in range(L)]
            S = scale * Q[:, h, :] @ K[:, h // G, :].T
            S = np.where(keep, S, -np.inf)
            for i in range(c):
                if not keep[i].any():
                    continue
                m = S[i].max()
                e = np.exp(S[i] - m)
                out[t0 + i, h] = e @ V[:, h // G, :] / e.sum()
                lse[t0 + i, h] = m + np.log(e.sum())
    return out, lse


@pytest.mark.parametrize("causal,kind", [(False, None), (False, "2d"), (True, "4d_heads"),
                                         (False, "4d_bcast")])
def test_dense_brute_force(causal, kind):
    batch = W.make_batch([0, 45, 130], [33, 1, 20], 4, 2, 64, 16, seed=69)
    mask = None if kind is None else W.random_mask(batch, kind, seed=70, keep=0.7)
    _, kp, vp, out, lse = oracle.run_batch(batch, causal=causal, mask=mask)
    ref_o, ref_l = dense_masked(batch, kp, vp, causal, mask)
    np.testing.assert_allclose(out, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_l, rtol=0, atol=1e-12)


def test_window_needs_causal():
    batch = W.make_batch([10], [5], 2, 1, 64, 16, seed=71, window=4)
    with pytest.raises(oracle.OracleError) as e:
        oracle.run_batch(batch, causal=False)
    assert e.value.code == oracle.ERR_INVALID_ARG


def test_keys_past_mask_extent_are_masked():
    batch = W.make_batch([40, 8], [10, 30], 4, 2, 64, 16, seed=72)
    full = W.random_mask(batch, "2d", seed=73, keep=0.8)
    short = full[:, :32].copy()
    padded = full.copy()
    padded[:, 32:] = False
    for causal in (True, False):
        _, _, _, o1, l1 = oracle.run_batch(batch, causal=causal, mask=short)
        _, _, _, o2, l2 = oracle.run_batch(batch, causal=causal, mask=padded)
        np.testing.assert_array_equal(o1, o2)
        np.testing.assert_array_equal(l1, l2)
