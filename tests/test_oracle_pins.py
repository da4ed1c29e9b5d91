"""Pins for the FP64 oracle: each check ties it to something other than itself.

* the zero-score worked example printed by AReno PR #642 ("What does this PR
  do?") -- a golden fixture;
* closed forms: Q = 0 with V_j = j gives the mean of the visible positions,
  and a window of one key gives V_p exactly;
* invariants: chunk-partition invariance (AReno PR #642 "How was it tested?":
  one-token chunks, 128/65/1 partitions), page-table permutation / padding /
  page-size invariance, GQA equal to MHA with replicated KV heads, the
  log-sum-exp merge of a prefix part and a chunk part;
* brute force: a dense numpy softmax over an explicit bottom-right mask,
  gathered through the page list by list expansion (a different route from the
  oracle's division-based slot formula);
* kv_append against numpy fancy-index assignment with a sentinel pool.

A plausible mistake in the oracle (top-left instead of bottom-right alignment,
an off-by-one window edge, a transposed page index, a wrong GQA head map, a
missing scale) fails at least one of these.
"""
import json
import os

import numpy as np
import pytest

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- helpers
def expand_slots(kv_indptr, kv_indices, b, page_size, length):
    """Logical key -> physical slot for sequence b by expanding its page list."""
    pages = kv_indices[kv_indptr[b]:kv_indptr[b + 1]]
    slots = []
    for pg in pages:
        if len(slots) >= length:
            break
        slots.extend(int(pg) * page_size + o for o in range(page_size))
    return np.asarray(slots[:length], dtype=np.int64)


def append_by_numpy(batch, k_pool, v_pool):
    """Scatter the chunk's K/V with numpy fancy indexing (independent of the oracle)."""
    for b in range(batch.batch):
        P = int(batch.prefix_lens[b])
        c = int(batch.chunk_lens[b])
        s = expand_slots(batch.kv_indptr, batch.kv_indices, b, batch.page_size, P + c)[P:P + c]
        t0 = int(batch.qo_indptr[b])
        k_pool[s] = batch.k_new[t0:t0 + c]
        v_pool[s] = batch.v_new[t0:t0 + c]


def dense_reference(batch, k_pool, v_pool):
    """Dense softmax attention with an explicit [c, L] bottom-right mask, float64."""
    Hq, Hkv, D = batch.n_q_heads, batch.n_kv_heads, batch.head_dim
    G = Hq // Hkv
    scale = batch.sm_scale if batch.sm_scale > 0 else 1.0 / np.sqrt(D)
    out = np.zeros((batch.total_q, Hq, D))
    lse = np.zeros((batch.total_q, Hq))
    for b in range(batch.batch):
        P, c = int(batch.prefix_lens[b]), int(batch.chunk_lens[b])
        L = P + c
        if c == 0:
            continue
        s = expand_slots(batch.kv_indptr, batch.kv_indices, b, batch.page_size, L)
        K = W.bf16_to_f32(k_pool[s]).astype(np.float64)          # [L, Hkv, D]
        V = W.bf16_to_f32(v_pool[s]).astype(np.float64)
        t0 = int(batch.qo_indptr[b])
        Q = W.bf16_to_f32(batch.q[t0:t0 + c]).astype(np.float64)  # [c, Hq, D]
        pos = P + np.arange(c)[:, None]
        key = np.arange(L)[None, :]
        mask = key <= pos
        if batch.window > 0:
            mask &= key > pos - batch.window
        for h in range(Hq):
            g = h // G
            S = scale * Q[:, h, :] @ K[:, g, :].T
            S = np.where(mask, S, -np.inf)
            m = S.max(axis=1, keepdims=True)
            E = np.exp(S - m)
            Z = E.sum(axis=1, keepdims=True)
            out[t0:t0 + c, h, :] = (E / Z) @ V[:, g, :]
            lse[t0:t0 + c, h] = (m + np.log(Z))[:, 0]
    return out, lse


def run_steps(steps):
    """Serve a prompt chunk by chunk: append each chunk, then attend."""
    outs, lses = [], []
    for st in steps:
        loc = oracle.out_cache_loc(st.qo_indptr, st.kv_indptr, st.kv_indices, st.prefix_lens,
                                   st.page_size, st.num_pages)
        oracle.kv_append(st.k_new, st.v_new, loc, st.k_pool, st.v_pool)
        o, l = oracle.paged_extend_attn(st.q, st.qo_indptr, st.kv_indptr, st.kv_indices,
                                        st.prefix_lens, st.k_pool, st.v_pool, st.page_size,
                                        st.n_q_heads, st.n_kv_heads, st.head_dim, st.window,
                                        st.sm_scale)
        outs.append(o)
        lses.append(l)
    return np.concatenate(outs), np.concatenate(lses)


def prompt_steps(q, k, v, chunks, page_size, n_q_heads, n_kv_heads, head_dim, window=0,
                 sm_scale=0.0, perm_seed=3, slack=2, pad=0):
    """Split one prompt (q/k/v bf16 bits, [T, H, D]) into chunk steps over a
    shared shuffled pool."""
    T = q.shape[0]
    assert sum(chunks) == T
    need = -(-T // page_size)
    rng = np.random.default_rng(perm_seed)
    num_pages = need + slack
    pages = rng.permutation(num_pages)[:need].astype(np.int32)
    k_pool = np.full((num_pages * page_size, n_kv_heads, head_dim), 0x7FC0, np.uint16)
    v_pool = k_pool.copy()
    steps, start = [], 0
    for c in chunks:
        L = start + c
        npg = -(-L // page_size)
        idx = np.concatenate([pages[:npg], np.full(pad, -1, np.int32)]).astype(np.int32)
        steps.append(W.Batch(
            name="prompt step", n_q_heads=n_q_heads, n_kv_heads=n_kv_heads, head_dim=head_dim,
            page_size=page_size, window=window, sm_scale=sm_scale,
            qo_indptr=np.array([0, c], np.int32), prefix_lens=np.array([start], np.int32),
            kv_indptr=np.array([0, idx.shape[0]], np.int32), kv_indices=idx,
            num_pages=num_pages, q=q[start:L], k_new=k[start:L], v_new=v[start:L],
            k_pool=k_pool, v_pool=v_pool))
        start = L
    return steps


def random_prompt(T, Hq, Hkv, D, seed):
    rng = np.random.default_rng(seed)
    f = lambda h: W.bf16_bits(rng.standard_normal((T, h, D), dtype=np.float32))
    return f(Hq), f(Hkv), f(Hkv)


# -------------------------------------------------------------------- pins
def test_zero_score_golden():
    g = json.load(open(os.path.join(GOLDEN, "zero_score.json")))
    for ps in (1, 2, 3, 16):
        steps = W.zero_score_steps(page_size=ps, chunks=tuple(g["chunks"]))
        out, lse = run_steps(steps)
        rows = out[:, 0, :]
        np.testing.assert_allclose(rows, np.broadcast_to(
            np.asarray(g["expected_rows"])[:, None], rows.shape), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[:, 0], np.log(np.arange(1, 5)), atol=1e-12)


def test_zero_score_chunk_local_reading_is_rejected():
    """Treating the second chunk as a fresh prompt (no cached prefix) gives the
    wrong numbers the page prints; the golden values tell the two apart."""
    g = json.load(open(os.path.join(GOLDEN, "zero_score.json")))
    steps = W.zero_score_steps(page_size=2, chunks=(2, 2))
    run_steps(steps[:1])
    st = steps[1]
    # keys 2,3 relabelled as a fresh 2-token prompt at positions 0,1
    fresh = W.Batch(**{**st.__dict__, "prefix_lens": np.array([0], np.int32),
                       "kv_indices": st.kv_indices[1:2].copy(),
                       "kv_indptr": np.array([0, 1], np.int32)})
    out, _ = run_steps([fresh])
    assert np.allclose(out[:, 0, 0], g["wrong_chunk_local_rows"][2:])
    assert not np.allclose(out[:, 0, 0], g["expected_rows"][2:])


@pytest.mark.parametrize("page_size", [1, 3, 16, 64])
@pytest.mark.parametrize("window", [0, 1, 5, 40])
def test_position_mean_closed_form(page_size, window):
    """Q = 0 and V_j = j (exact in bf16 for j <= 256): each row's output is the
    mean of its visible positions, (lo + p) / 2, and lse = ln(p - lo + 1)."""
    T, Hq, Hkv, D = 200, 4, 2, 16
    q = np.zeros((T, Hq, D), np.uint16)
    _, k, _ = random_prompt(T, Hq, Hkv, D, seed=11)
    v = W.bf16_bits(np.broadcast_to(np.arange(T, dtype=np.float32)[:, None, None],
                                    (T, Hkv, D)))
    steps = prompt_steps(q, k, v, [37, 1, 1, 90, 71], page_size, Hq, Hkv, D, window=window,
                         pad=2)
    out, lse = run_steps(steps)
    p = np.arange(T, dtype=np.float64)
    lo = np.maximum(0, p - window + 1) if window > 0 else np.zeros(T)
    want = (lo + p) / 2
    np.testing.assert_allclose(out, np.broadcast_to(want[:, None, None], out.shape),
                               atol=1e-9, rtol=0)
    np.testing.assert_allclose(lse, np.broadcast_to(np.log(p - lo + 1)[:, None], lse.shape),
                               atol=1e-12)


def test_single_visible_key():
    """Window 1: a row sees only its own key, so out = V_p exactly and
    lse = sm_scale * q . k_p."""
    T, Hq, Hkv, D = 70, 2, 1, 64
    q, k, v = random_prompt(T, Hq, Hkv, D, seed=5)
    steps = prompt_steps(q, k, v, [30, 40], 16, Hq, Hkv, D, window=1, sm_scale=0.125)
    out, lse = run_steps(steps)
    vf = W.bf16_to_f32(v).astype(np.float64)
    for h in range(Hq):
        np.testing.assert_array_equal(out[:, h, :], vf[:, 0, :])
    dots = (W.bf16_to_f32(q).astype(np.float64) * W.bf16_to_f32(k).astype(np.float64)).sum(-1)
    np.testing.assert_allclose(lse, 0.125 * dots, atol=1e-12)


def test_first_row_of_fresh_prompt_sees_itself():
    T, Hq, Hkv, D = 9, 2, 2, 64
    q, k, v = random_prompt(T, Hq, Hkv, D, seed=6)
    out, _ = run_steps(prompt_steps(q, k, v, [9], 4, Hq, Hkv, D))
    np.testing.assert_array_equal(out[0], W.bf16_to_f32(v[0]).astype(np.float64))


@pytest.mark.parametrize("chunks", [[300], [1] * 300, [128, 65, 7, 1, 99],
                                    [65, 128, 1, 7, 1, 98]])
def test_chunk_partition_invariance(chunks):
    T, Hq, Hkv, D = 300, 4, 2, 64
    q, k, v = random_prompt(T, Hq, Hkv, D, seed=21)
    ref, ref_lse = run_steps(prompt_steps(q, k, v, [300], 16, Hq, Hkv, D))
    out, lse = run_steps(prompt_steps(q, k, v, chunks, 16, Hq, Hkv, D))
    np.testing.assert_allclose(out, ref, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse, ref_lse, atol=1e-12, rtol=0)


@pytest.mark.parametrize("window", [0, 50])
def test_page_layout_invariance(window):
    """Physical placement must not matter: permuted pools, page sizes 1/16/64,
    and -1 padding after the needed pages give bit-identical results."""
    T, Hq, Hkv, D = 260, 4, 1, 64
    q, k, v = random_prompt(T, Hq, Hkv, D, seed=31)
    chunks = [100, 1, 159]
    ref = None
    for ps, seed, pad in [(16, 1, 0), (16, 2, 3), (1, 3, 0), (64, 4, 5), (3, 5, 1)]:
        o, l = run_steps(prompt_steps(q, k, v, chunks, ps, Hq, Hkv, D, window=window,
                                      perm_seed=seed, pad=pad))
        if ref is None:
            ref = (o, l)
        else:
            np.testing.assert_array_equal(o, ref[0])
            np.testing.assert_array_equal(l, ref[1])


@pytest.mark.parametrize("window", [0, 33])
def test_dense_brute_force(window):
    batch = W.make_batch([0, 37, 5, 64], [5, 40, 1, 17], 4, 2, 32, 8, seed=41, window=window,
                         sm_scale=0.2, pad_to_pages=16)
    kp, vp = batch.k_pool.copy(), batch.v_pool.copy()
    append_by_numpy(batch, kp, vp)
    want, want_lse = dense_reference(batch, kp, vp)
    _, _, _, out, lse = oracle.run_batch(batch)
    np.testing.assert_allclose(out, want, atol=1e-11, rtol=0)
    np.testing.assert_allclose(lse, want_lse, atol=1e-11, rtol=0)


def test_tiny_case_against_dense():
    batch = W.tiny_case()
    kp, vp = batch.k_pool.copy(), batch.v_pool.copy()
    append_by_numpy(batch, kp, vp)
    want, want_lse = dense_reference(batch, kp, vp)
    _, _, _, out, lse = oracle.run_batch(batch)
    np.testing.assert_allclose(out, want, atol=1e-11, rtol=0)
    np.testing.assert_allclose(lse, want_lse, atol=1e-11, rtol=0)


def test_default_scale_is_inverse_sqrt_head_dim():
    batch = W.make_batch([3], [4], 2, 1, 64, 4, seed=43)
    b2 = W.Batch(**{**batch.__dict__, "sm_scale": 1.0 / 8.0})
    _, _, _, o1, l1 = oracle.run_batch(batch)
    _, _, _, o2, l2 = oracle.run_batch(b2)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_gqa_equals_mha_with_replicated_heads():
    T, Hq, Hkv, D = 90, 8, 2, 32
    q, k, v = random_prompt(T, Hq, Hkv, D, seed=51)
    k_rep = np.repeat(k, Hq // Hkv, axis=1)
    v_rep = np.repeat(v, Hq // Hkv, axis=1)
    o1, l1 = run_steps(prompt_steps(q, k, v, [40, 50], 16, Hq, Hkv, D))
    o2, l2 = run_steps(prompt_steps(q, k_rep, v_rep, [40, 50], 16, Hq, Hq, D))
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_lse_merge_of_prefix_and_chunk():
    """out over [0, p] equals the lse-weighted merge of out over [0, P) and
    out over [P, p] -- the identity split-KV combining rests on."""
    T, Hq, Hkv, D, P = 120, 2, 1, 64, 70
    q, k, v = random_prompt(T, Hq, Hkv, D, seed=61)
    full, full_lse = run_steps(prompt_steps(q, k, v, [P, T - P], 16, Hq, Hkv, D))
    for p in (P, P + 1, P + 17, T - 1):
        # part A: keys [0, P) seen by this row's query placed at position P-1
        qa = k.copy()[:P].copy()
        qa_q = q[:P].copy()
        qa_q[P - 1] = q[p]
        oa, la = run_steps(prompt_steps(qa_q, qa, v[:P], [P], 16, Hq, Hkv, D))
        oa, la = oa[P - 1], la[P - 1]
        # part B: keys [P, p] relabelled 0..p-P, query at the last of them
        n = p - P + 1
        qb_q = q[P:p + 1].copy()
        qb_q[n - 1] = q[p]
        ob, lb = run_steps(prompt_steps(qb_q, k[P:p + 1], v[P:p + 1], [n], 16, Hq, Hkv, D))
        ob, lb = ob[n - 1], lb[n - 1]
        lse = np.logaddexp(la, lb)
        merged = np.exp(la - lse)[:, None] * oa + np.exp(lb - lse)[:, None] * ob
        np.testing.assert_allclose(merged, full[p], atol=1e-12, rtol=0)
        np.testing.assert_allclose(lse, full_lse[p], atol=1e-12, rtol=0)


def test_row_selection_matches_full():
    batch = W.stress_case(16, 64, batch=6, max_prefix=300)
    _, _, _, out, lse = oracle.run_batch(batch)
    rng = np.random.default_rng(0)
    tok = rng.integers(0, batch.total_q, size=40)
    head = rng.integers(0, batch.n_q_heads, size=40).astype(np.int32)
    _, _, _, o2, l2 = oracle.run_batch(batch, rows=(tok, head))
    np.testing.assert_array_equal(o2, out[tok, head])
    np.testing.assert_array_equal(l2, lse[tok, head])


# ------------------------------------------------------ append and slots
@pytest.mark.parametrize("page_size", [1, 16, 64])
def test_out_cache_loc_and_append(page_size):
    batch = W.make_batch([0, 13, 64, 200], [5, 40, 1, 77], 4, 2, 16, page_size, seed=71,
                         pad_to_pages=400 // page_size + 2)
    loc = oracle.out_cache_loc(batch.qo_indptr, batch.kv_indptr, batch.kv_indices,
                               batch.prefix_lens, batch.page_size, batch.num_pages)
    want = np.concatenate([
        expand_slots(batch.kv_indptr, batch.kv_indices, b, page_size,
                     int(batch.kv_lens[b]))[int(batch.prefix_lens[b]):]
        for b in range(batch.batch)])
    np.testing.assert_array_equal(loc, want)
    sentinel = np.full_like(batch.k_pool, 0xBEEF)
    kp, vp = sentinel.copy(), sentinel.copy()
    oracle.kv_append(batch.k_new, batch.v_new, loc, kp, vp)
    kw, vw = sentinel.copy(), sentinel.copy()
    kw[want] = batch.k_new
    vw[want] = batch.v_new
    np.testing.assert_array_equal(kp, kw)
    np.testing.assert_array_equal(vp, vw)
    untouched = np.ones(kp.shape[0], bool)
    untouched[want] = False
    assert (kp[untouched] == 0xBEEF).all() and (vp[untouched] == 0xBEEF).all()


def test_mid_page_append_continues_in_last_page():
    """A prefix of 13 tokens with page_size 16 leaves 3 free slots in the last
    page: the first three new tokens land there, the rest in the next page."""
    batch = W.make_batch([13], [6], 1, 1, 16, 16, seed=72)
    loc = oracle.out_cache_loc(batch.qo_indptr, batch.kv_indptr, batch.kv_indices,
                               batch.prefix_lens, 16, batch.num_pages)
    p0, p1 = int(batch.kv_indices[0]), int(batch.kv_indices[1])
    np.testing.assert_array_equal(loc, [p0 * 16 + 13, p0 * 16 + 14, p0 * 16 + 15,
                                        p1 * 16, p1 * 16 + 1, p1 * 16 + 2])


def test_bad_pages_are_errors():
    batch = W.make_batch([20], [10], 2, 1, 16, 16, seed=73)
    bad = batch.kv_indices.copy()
    bad[1] = -1
    with pytest.raises(oracle.OracleError) as e:
        oracle.out_cache_loc(batch.qo_indptr, batch.kv_indptr, bad, batch.prefix_lens, 16,
                             batch.num_pages)
    assert e.value.code == oracle.ERR_BAD_INDEX
    bad[1] = batch.num_pages
    with pytest.raises(oracle.OracleError):
        oracle.paged_extend_attn(batch.q, batch.qo_indptr, batch.kv_indptr, bad,
                                 batch.prefix_lens, batch.k_pool, batch.v_pool, 16, 2, 1, 16)
    with pytest.raises(oracle.OracleError):
        oracle.kv_append(batch.k_new, batch.v_new, np.full(10, batch.pool_slots, np.int64),
                         batch.k_pool.copy(), batch.v_pool.copy())


def test_empty_chunks_and_empty_batch():
    batch = W.make_batch([5, 0, 9], [0, 3, 0], 2, 1, 16, 4, seed=74)
    _, _, _, out, lse = oracle.run_batch(batch)
    assert out.shape == (3, 2, 16)
    empty = W.make_batch([], [], 2, 1, 16, 4, seed=75)
    _, _, _, out, lse = oracle.run_batch(empty)
    assert out.shape == (0, 2, 16) and lse.shape == (0, 2)


def test_generator_is_deterministic():
    a, b = W.tiny_case(), W.tiny_case()
    for f in ("q", "k_new", "v_new", "k_pool", "kv_indices", "qo_indptr", "prefix_lens"):
        np.testing.assert_array_equal(getattr(a, f), getattr(b, f))
    m = W.mixed_batch(decode_max=256)
    assert m.batch == 34 and m.total_q == 4097 + 31
    assert list(m.chunk_lens[:3]) == [2048, 2048, 1] and list(m.prefix_lens[:3]) == [0, 2048, 4096]
    s = W.stress_case(16, 4096, batch=16, max_prefix=2048)
    assert ((s.prefix_lens % 16) > 0).all()
    assert set(np.unique(s.chunk_lens)).issubset({1, 7, 65, 128})
