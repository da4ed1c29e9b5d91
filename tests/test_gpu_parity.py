"""GPU parity: the CUDA path (through the C ABI) against the FP64 oracle.

Small cases are compared element by element over every row; the full-size
workloads on sampled rows (every head of the edge rows of the first
sequences, random rows elsewhere).  out_cache_loc and the appended pools must
be bit-exact; bf16 outputs within max-abs 2e-2 / mean-abs 2e-3; lse within
1e-3.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from helpers import (assert_close, bf16_tensor_bits, bf16_tensor_to_f64, run_gpu,
                     sample_rows, to_device)

pytestmark = pytest.mark.gpu


def full_parity(batch, what=""):
    loc, d, out, lse = run_gpu(batch)
    loc_ref, kp_ref, vp_ref, out_ref, lse_ref = oracle.run_batch(batch)
    np.testing.assert_array_equal(loc.cpu().numpy(), loc_ref)
    np.testing.assert_array_equal(bf16_tensor_bits(d["k_pool"]), kp_ref)
    np.testing.assert_array_equal(bf16_tensor_bits(d["v_pool"]), vp_ref)
    return assert_close(bf16_tensor_to_f64(out), lse.cpu().numpy().astype(np.float64), out_ref,
                        lse_ref, what or batch.name)


def sampled_parity(batch, n_random=256, what=""):
    loc, d, out, lse = run_gpu(batch)
    loc_ref = oracle.out_cache_loc(batch.qo_indptr, batch.kv_indptr, batch.kv_indices,
                                   batch.prefix_lens, batch.page_size, batch.num_pages)
    np.testing.assert_array_equal(loc.cpu().numpy(), loc_ref)
    # the appended pools, read back from the GPU, are the oracle's inputs
    kp = bf16_tensor_bits(d["k_pool"])
    vp = bf16_tensor_bits(d["v_pool"])
    np.testing.assert_array_equal(kp[loc_ref], batch.k_new)
    np.testing.assert_array_equal(vp[loc_ref], batch.v_new)
    untouched = np.ones(kp.shape[0], bool)
    untouched[loc_ref] = False
    assert (kp[untouched] == batch.k_pool[untouched]).all()
    tok, head = sample_rows(batch, n_random)
    out_ref, lse_ref = oracle.paged_extend_attn(
        batch.q, batch.qo_indptr, batch.kv_indptr, batch.kv_indices, batch.prefix_lens, kp, vp,
        batch.page_size, batch.n_q_heads, batch.n_kv_heads, batch.head_dim, batch.window,
        batch.sm_scale, rows=(tok, head))
    o = bf16_tensor_to_f64(out)[tok, head]
    l = lse.cpu().numpy().astype(np.float64)[tok, head]
    return assert_close(o, l, out_ref, lse_ref, what or batch.name)


# ----------------------------------------------------------------- workloads
def test_tiny_case():
    full_parity(W.tiny_case())


@pytest.mark.parametrize("chunks", [(2, 2), (40, 40), (100, 28)])
def test_zero_score_on_gpu(chunks):
    """AReno PR #642's zero-score regression: Q = 0, V_j = 2j + 1; row i of the
    prompt sees keys 0..i, so it gives i + 1 (the 4-token prompt as two 2-token
    chunks gives 1, 2, 3, 4, not 1, 2, 5, 6).  Small chunks run on the row
    kernel, larger ones on the tensor cores."""
    for ps in (1, 2, 16):
        steps = W.zero_score_steps(page_size=ps, chunks=chunks)
        d0 = to_device(steps[0])
        pools = (d0["k_pool"], d0["v_pool"])
        rows = []
        for st in steps:
            d = to_device(st)
            d["k_pool"], d["v_pool"] = pools
            _, _, out, lse = run_gpu(st, d)
            rows.append(bf16_tensor_to_f64(out)[:, 0, :])
        rows = np.concatenate(rows)
        want = np.arange(1, sum(chunks) + 1, dtype=np.float64)[:, None]
        np.testing.assert_array_equal(rows, np.repeat(want, rows.shape[1], axis=1))


def test_gqa_prefill_reduced():
    full_parity(W.gqa_prefill(batch=3, max_prefix=700, chunk=300))


def test_mixed_reduced():
    full_parity(W.mixed_batch(prompt=700, chunk=300, n_decode=9, decode_max=1500))


@pytest.mark.parametrize("ps,window", [(1, 4096), (1, 0), (16, 4096), (16, 0)])
def test_stress_reduced(ps, window):
    full_parity(W.stress_case(ps, window, batch=16, max_prefix=2000))


@pytest.mark.parametrize("name", ["gqa_prefill", "mixed", "stress_ps1_w4096", "stress_ps1_w0",
                                  "stress_ps16_w4096", "stress_ps16_w0"])
def test_full_size_sampled(name):
    sampled_parity(W.config_by_name(name), n_random=256)


def test_long_context_sampled():
    sampled_parity(W.long_context(), n_random=128)


# ---------------------------------------------------------------- edge cases
@pytest.mark.parametrize("ps", [1, 2, 3, 8, 16, 32, 64, 128, 256])
def test_page_sizes(ps):
    b = W.make_batch([0, 5, 130, 257, 1000], [37, 200, 1, 129, 64], 8, 2, 64, ps, seed=ps,
                     pad_to_pages=1100 // ps + 3)
    full_parity(b, f"page_size {ps}")


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 4), (16, 4), (32, 4), (64, 2), (16, 1), (12, 4)])
@pytest.mark.parametrize("d", [64, 128])
def test_group_sizes(hq, hkv, d):
    b = W.make_batch([0, 77, 300], [150, 1, 90], hq, hkv, d, 16, seed=hq * 10 + hkv + d)
    full_parity(b, f"Hq={hq} Hkv={hkv} D={d}")


@pytest.mark.parametrize("window", [1, 2, 127, 128, 129, 300])
def test_windows(window):
    b = W.make_batch([0, 200, 513, 40], [260, 129, 1, 3], 8, 2, 128, 16, seed=window,
                     window=window)
    full_parity(b, f"window {window}")


@pytest.mark.parametrize("case", ["mixed", "decode", "prefill"])
def test_host_hint_is_bit_identical(case):
    """With and without the host copy of qo_indptr the same kernels do the
    work (the hint only skips launches that have none): identical bits."""
    if case == "mixed":
        b = W.mixed_batch(prompt=700, chunk=300, n_decode=9, decode_max=1500)
    elif case == "decode":
        b = W.make_batch([5, 900, 3000, 40], [1, 1, 2, 1], 16, 4, 128, 64, seed=30)
    else:
        b = W.make_batch([0, 300], [200, 77], 16, 4, 128, 16, seed=31)
    res = []
    for hint in (True, False):
        _, _, out, lse = run_gpu(b, host_hint=hint)
        res.append((bf16_tensor_bits(out), lse.cpu().numpy()))
    np.testing.assert_array_equal(res[0][0], res[1][0])
    np.testing.assert_array_equal(res[0][1], res[1][1])
    full_parity(b, f"hinted {case}")


@pytest.mark.parametrize("n,ps,window", [(1, 64, 0), (31, 16, 0), (300, 1, 0), (512, 64, 700),
                                          (513, 16, 0)])
def test_self_planned_decode_is_bit_identical(n, ps, window):
    """A decode-only call with the host copy of qo_indptr and at most 512
    sequences is planned inside the row kernel (no planner launch); without
    the copy the planner kernel plans it.  Both give identical bits, also
    with zero-length chunks, two-row chunks and a window (513 sequences:
    the planner both times)."""
    rng = np.random.default_rng(n + ps)
    P = rng.integers(1, 5000 if n < 100 else 1500, size=n)
    C = rng.choice([0, 1, 1, 1, 2], size=n)
    C[0] = 1  # at least one row
    hq, hkv, d = (16, 4, 128) if n < 100 else (8, 2, 64)
    b = W.make_batch(P, C, hq, hkv, d, ps, seed=60 + n, window=window)
    res = []
    for hint in (True, False):
        _, _, out, lse = run_gpu(b, host_hint=hint)
        res.append((bf16_tensor_bits(out), lse.cpu().numpy()))
    np.testing.assert_array_equal(res[0][0], res[1][0])
    np.testing.assert_array_equal(res[0][1], res[1][1])
    sampled_parity(b, n_random=128, what=f"self-planned decode n={n} ps={ps} W={window}")


def test_decode_rows_many_splits():
    """A few very long decode rows and many short ones: the long groups span
    many row-kernel CTAs (many partial slots), the short ones share a CTA."""
    rng = np.random.default_rng(12)
    P = [60000, 45000] + list(rng.integers(1, 300, size=40))
    b = W.make_batch(P, [1] * len(P), 8, 2, 128, 16, seed=32)
    full_parity(b, "many splits")


@pytest.mark.parametrize("ps", [8, 24, 48, 112])
def test_decode_rows_page_windows(ps):
    """Long decode rows over small and odd page sizes: the row kernel reads
    page ids through a moving window of page-table entries, with tiles that
    straddle its halves when the page size does not divide 128; some rows
    start past key 0 (sliding window) and some are split across CTAs."""
    rng = np.random.default_rng(ps)
    P = [9000, 7001, 3000] + list(rng.integers(1, 2500, size=9))
    for window in (0, 2000):
        b = W.make_batch(P, [1] * len(P), 16, 4, 128, ps, seed=50 + ps, window=window)
        full_parity(b, f"decode rows, page_size {ps}, window {window}")


def test_decode_only_long():
    """Many decode rows with long KV: split-KV pieces and the combine."""
    b = W.make_batch(list(np.random.default_rng(3).integers(1, 9000, size=12)), [1] * 12, 16, 4,
                     128, 64, seed=33)
    full_parity(b, "decode rows")


def test_small_chunks_decode_path():
    """chunk_len * G <= 16 goes to the row kernel: c in {1, 2, 4} with G = 4."""
    b = W.make_batch([100, 2000, 5, 0], [1, 2, 4, 3], 16, 4, 128, 16, seed=34, window=1000)
    full_parity(b, "small chunks")


def test_empty_and_zero_length_chunks():
    import paged_chunked_prefill_gb300 as pcp
    b = W.make_batch([5, 0, 9, 70], [0, 3, 0, 130], 4, 2, 64, 4, seed=35)
    full_parity(b, "zero-length chunks")
    e = W.make_batch([], [], 4, 2, 64, 4, seed=36)
    loc, d, out, lse = run_gpu(e)
    assert out.shape == (0, 4, 64) and lse.shape == (0, 4) and loc.numel() == 0


def test_default_scale():
    b = W.make_batch([10, 300], [200, 50], 8, 2, 128, 16, seed=37, sm_scale=0.0)
    full_parity(b, "default scale")


def test_garbage_pool_tail_does_not_leak():
    """Slots past a sequence's end inside its last page (and every unused slot)
    hold NaN: masked keys must not leak into the outputs."""
    b = W.make_batch([13, 0, 250], [170, 45, 1], 8, 2, 128, 64, seed=38)
    nan = np.uint16(0x7FC0)
    used = np.zeros(b.pool_slots, bool)
    for i in range(b.batch):
        pages = b.kv_indices[b.kv_indptr[i]:b.kv_indptr[i + 1]]
        L = int(b.kv_lens[i])
        slots = np.concatenate([p * b.page_size + np.arange(b.page_size) for p in pages])[:L]
        used[slots] = True
    b.k_pool[~used] = nan
    b.v_pool[~used] = nan
    full_parity(b, "NaN tails")


def test_page_layout_bit_identical():
    """The same logical K/V through different page sizes and permutations gives
    bit-identical GPU outputs (tiles follow logical positions)."""
    outs = []
    rng = np.random.default_rng(5)
    P, C = [0, 300, 1500], [400, 64, 1]
    Hq, Hkv, D = 16, 4, 128
    L = [p + c for p, c in zip(P, C)]
    q = W.bf16_bits(rng.standard_normal((sum(C), Hq, D), dtype=np.float32))
    kv = [W.bf16_bits(rng.standard_normal((l, Hkv, D), dtype=np.float32)) for l in L]
    vv = [W.bf16_bits(rng.standard_normal((l, Hkv, D), dtype=np.float32)) for l in L]
    for ps, seed in [(16, 1), (16, 2), (64, 3), (1, 4), (128, 5)]:
        b = W.make_batch(P, C, Hq, Hkv, D, ps, seed=seed)
        b.q[:] = q
        for i in range(3):
            pages = b.kv_indices[b.kv_indptr[i]:b.kv_indptr[i + 1]]
            slots = np.concatenate([p * ps + np.arange(ps) for p in pages])[:L[i]]
            b.k_pool[slots[:P[i]]] = kv[i][:P[i]]
            b.v_pool[slots[:P[i]]] = vv[i][:P[i]]
            t0 = int(b.qo_indptr[i])
            b.k_new[t0:t0 + C[i]] = kv[i][P[i]:]
            b.v_new[t0:t0 + C[i]] = vv[i][P[i]:]
        _, _, out, lse = run_gpu(b)
        outs.append((bf16_tensor_bits(out), lse.cpu().numpy()))
    for o, l in outs[1:]:
        np.testing.assert_array_equal(o, outs[0][0])
        np.testing.assert_array_equal(l, outs[0][1])


def test_chunk_partition_invariance_gpu():
    """Serving a prompt in chunks (including 1-token chunks) matches serving it
    in one chunk, within tolerance."""
    import paged_chunked_prefill_gb300 as pcp
    rng = np.random.default_rng(9)
    T, Hq, Hkv, D, ps = 400, 8, 2, 128, 16
    q = W.bf16_bits(rng.standard_normal((T, Hq, D), dtype=np.float32))
    k = W.bf16_bits(rng.standard_normal((T, Hkv, D), dtype=np.float32))
    v = W.bf16_bits(rng.standard_normal((T, Hkv, D), dtype=np.float32))
    results = []
    for chunks in ([400], [128, 65, 7, 1, 199], [1] * 5 + [395]):
        b0 = W.make_batch([0], [T], Hq, Hkv, D, ps, seed=77)
        d = to_device(b0)
        outs, lses, start = [], [], 0
        for c in chunks:
            L = start + c
            npg = -(-L // ps)
            st = W.Batch(**{**b0.__dict__, "qo_indptr": np.array([0, c], np.int32),
                            "prefix_lens": np.array([start], np.int32),
                            "kv_indptr": np.array([0, npg], np.int32),
                            "kv_indices": b0.kv_indices[:npg].copy(), "q": q[start:L],
                            "k_new": k[start:L], "v_new": v[start:L]})
            ds = to_device(st)
            ds["k_pool"], ds["v_pool"] = d["k_pool"], d["v_pool"]
            _, _, out, lse = run_gpu(st, ds)
            outs.append(bf16_tensor_to_f64(out))
            lses.append(lse.cpu().numpy().astype(np.float64))
            start = L
        results.append((np.concatenate(outs), np.concatenate(lses)))
    for o, l in results[1:]:
        assert_close(o, l, results[0][0], results[0][1], "partition")


# ------------------------------------------------- fused slot mapping + append
@pytest.mark.parametrize("name", ["tiny", "mixed", "stress_ps1_w0", "stress_ps16_w4096",
                                  "gqa_prefill"])
def test_fused_append_bit_exact(name):
    """pcp_kv_append_paged: the slots and the appended pools equal the
    oracle's slot mapping and scatter bit for bit; slots no token names keep
    their contents."""
    import torch
    import paged_chunked_prefill_gb300 as pcp
    batch = W.config_by_name(name)
    d = to_device(batch)
    loc = torch.full((batch.total_q,), -7, dtype=torch.int64, device="cuda")
    pcp.kv_append_paged(d["qo_indptr"], d["kv_indptr"], d["kv_indices"], d["prefix_lens"],
                        batch.page_size, d["k_new"], d["v_new"], d["k_pool"], d["v_pool"],
                        out_cache_loc=loc)
    loc_ref = oracle.out_cache_loc(batch.qo_indptr, batch.kv_indptr, batch.kv_indices,
                                   batch.prefix_lens, batch.page_size, batch.num_pages)
    kp_ref, vp_ref = batch.k_pool.copy(), batch.v_pool.copy()
    oracle.kv_append(batch.k_new, batch.v_new, loc_ref, kp_ref, vp_ref)
    np.testing.assert_array_equal(loc.cpu().numpy(), loc_ref)
    np.testing.assert_array_equal(bf16_tensor_bits(d["k_pool"]), kp_ref)
    np.testing.assert_array_equal(bf16_tensor_bits(d["v_pool"]), vp_ref)


def test_fused_append_without_loc_then_attention():
    """The fused append with no out_cache_loc array, followed by attention:
    the same results as the separate slot mapping and append."""
    import torch
    import paged_chunked_prefill_gb300 as pcp
    batch = W.mixed_batch(prompt=700, chunk=300, n_decode=9, decode_max=3000)
    d = to_device(batch)
    pcp.kv_append_paged(d["qo_indptr"], d["kv_indptr"], d["kv_indices"], d["prefix_lens"],
                        batch.page_size, d["k_new"], d["v_new"], d["k_pool"], d["v_pool"])
    out, lse = pcp.paged_extend_attn(d["q"], d["qo_indptr"], d["kv_indptr"], d["kv_indices"],
                                     d["prefix_lens"], d["k_pool"], d["v_pool"],
                                     batch.page_size, batch.n_q_heads, batch.n_kv_heads,
                                     batch.head_dim, batch.window, batch.sm_scale)
    _, _, out2, lse2 = run_gpu(batch)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse2.view(torch.int32))


def test_fused_append_reports_bad_page():
    """A bad page id among a chunk's pages: PCP_ERR_BAD_INDEX, slot -1, that
    token not written, every other token appended."""
    import torch
    import paged_chunked_prefill_gb300 as pcp
    b = W.make_batch([10], [50], 8, 2, 64, 16, seed=41)
    bad = b.kv_indices.copy()
    bad[3] = -1          # keys 48..63: tokens 38..49 of the chunk
    b2 = W.Batch(**{**b.__dict__, "kv_indices": bad})
    d = to_device(b2)
    loc = torch.zeros(b.total_q, dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pcp.kv_append_paged(d["qo_indptr"], d["kv_indptr"], d["kv_indices"], d["prefix_lens"], 16,
                        d["k_new"], d["v_new"], d["k_pool"], d["v_pool"], out_cache_loc=loc,
                        dev_err=err)
    assert pcp.read_error(err) == pcp.Status.BAD_INDEX
    l = loc.cpu().numpy()
    pos = 10 + np.arange(50)
    assert (l[pos // 16 == 3] == -1).all()
    good = pos // 16 != 3
    np.testing.assert_array_equal(l[good], b.kv_indices[pos[good] // 16] * 16 + pos[good] % 16)
    kp = bf16_tensor_bits(d["k_pool"])
    np.testing.assert_array_equal(kp[l[good]], b.k_new[good])


# ------------------------------------------------------------------- errors
def test_bad_page_id_is_reported():
    import paged_chunked_prefill_gb300 as pcp
    b = W.make_batch([100], [50], 8, 2, 64, 16, seed=40)
    bad = b.kv_indices.copy()
    bad[2] = b.num_pages + 5   # a prefix page (keys 32..47)
    b2 = W.Batch(**{**b.__dict__, "kv_indices": bad})
    with pytest.raises(pcp.PCPError) as e:
        run_gpu(b2)
    assert e.value.status == pcp.Status.BAD_INDEX


def test_bad_chunk_page_reported_by_slot_mapping():
    import paged_chunked_prefill_gb300 as pcp
    b = W.make_batch([10], [50], 8, 2, 64, 16, seed=41)
    bad = b.kv_indices.copy()
    bad[-1] = -1
    d = to_device(W.Batch(**{**b.__dict__, "kv_indices": bad}))
    with pytest.raises(pcp.PCPError) as e:
        pcp.compute_out_cache_loc(d["qo_indptr"], d["kv_indptr"], d["kv_indices"],
                                  d["prefix_lens"], 16, b.num_pages)
    assert e.value.status == pcp.Status.BAD_INDEX


@pytest.mark.parametrize("last", [45, 55])
def test_device_qo_indptr_end_must_be_total_q(last):
    """Without the host copy, the planner checks on the device that
    qo_indptr[batch] equals total_q (the rows of q); a sequence that would
    run past total_q is skipped, so nothing is read or written out of range."""
    import paged_chunked_prefill_gb300 as pcp
    import torch
    b = W.make_batch([10, 60], [20, 30], 8, 2, 64, 16, seed=43)
    d = to_device(b)
    qo = torch.tensor([0, 20, last], dtype=torch.int32, device="cuda")
    with pytest.raises(pcp.PCPError) as e:
        pcp.paged_extend_attn(d["q"], qo, d["kv_indptr"], d["kv_indices"], d["prefix_lens"],
                              d["k_pool"], d["v_pool"], 16, 8, 2, 64)
    assert e.value.status == pcp.Status.INVALID_ARG


def test_host_errors_before_launch():
    import paged_chunked_prefill_gb300 as pcp
    import torch
    b = W.make_batch([10], [20], 8, 2, 64, 16, seed=42)
    d = to_device(b)
    tiny_ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(pcp.PCPError) as e:
        pcp.paged_extend_attn(d["q"], d["qo_indptr"], d["kv_indptr"], d["kv_indices"],
                              d["prefix_lens"], d["k_pool"], d["v_pool"], 16, 8, 2, 64,
                              workspace=tiny_ws)
    assert e.value.status == pcp.Status.WORKSPACE
    q96 = torch.zeros(20, 8, 96, dtype=torch.bfloat16, device="cuda")
    pool96 = torch.zeros(d["k_pool"].shape[0], 2, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pcp.PCPError) as e:
        pcp.paged_extend_attn(q96, d["qo_indptr"], d["kv_indptr"], d["kv_indices"],
                              d["prefix_lens"], pool96, pool96, 16, 8, 2, 96)
    assert e.value.status == pcp.Status.UNSUPPORTED
