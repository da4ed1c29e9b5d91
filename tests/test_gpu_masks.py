"""GPU parity of non-causal attention and boolean masks against the FP64
oracle (AstrAI attn_paged_prefill: `is_causal` and `mask`, True = keep).

The same kernels serve these calls: a causal flag changes each row's key
range and a mask adds a per-key test, on the tensor-core path and on the
split-KV row path.  Tolerances: bf16 out max-abs 2e-2 / mean-abs 2e-3, lse
1e-3; rows that see no key must give out = 0 and lse = -inf exactly.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from helpers import assert_close, bf16_tensor_to_f64, run_gpu

pytestmark = pytest.mark.gpu


def parity(batch, causal=True, mask=None, what=""):
    _, _, out, lse = run_gpu(batch, causal=causal, mask=mask)
    _, _, _, out_ref, lse_ref = oracle.run_batch(batch, causal=causal, mask=mask)
    o = bf16_tensor_to_f64(out)
    l = lse.cpu().numpy().astype(np.float64)
    empty = np.isneginf(lse_ref)
    assert (np.isneginf(l) == empty).all(), f"{what}: rows without keys differ"
    assert (o[empty] == 0).all()
    l = np.where(empty, 0.0, l)
    return assert_close(o, l, out_ref, np.where(empty, 0.0, lse_ref), what)


BATCHES = {
    # chunks on the tensor cores and decode-shaped rows, page sizes 16 / 1 / 64
    "mixed_ps16": lambda: W.make_batch([0, 300, 17, 900, 5], [200, 1, 129, 2, 64], 16, 4, 128,
                                       16, seed=81),
    "mixed_ps1": lambda: W.make_batch([40, 0, 333], [70, 3, 1], 8, 2, 64, 1, seed=82),
    "decode_ps64": lambda: W.make_batch([1000, 63, 4000, 128], [1, 1, 1, 1], 16, 4, 128, 64,
                                        seed=83),
}


@pytest.mark.parametrize("name", list(BATCHES))
def test_non_causal(name):
    parity(BATCHES[name](), causal=False, what=f"non-causal {name}")


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("kind", ["2d", "4d_bcast", "4d_heads", "4d_q1"])
@pytest.mark.parametrize("name", list(BATCHES))
def test_masks(name, kind, causal):
    b = BATCHES[name]()
    parity(b, causal=causal, mask=W.random_mask(b, kind, seed=84, keep=0.6),
           what=f"{name} {kind} causal={causal}")


def test_four_d_causal_mask_regression():
    """The pages' regression shape: one pure prefill request, a 4-D
    [1, 1, q, q] causal-pattern mask with causality off."""
    for q_len, (hq, hkv, d) in [(512, (32, 4, 128)), (1024, (32, 4, 128)), (256, (4, 2, 64))]:
        b = W.make_batch([0], [q_len], hq, hkv, d, 16, seed=q_len + d)
        m = np.tril(np.ones((q_len, q_len), bool))[None, None]
        parity(b, causal=False, mask=m, what=f"4-D causal mask q={q_len}")
        _, _, o1, l1 = run_gpu(b, causal=False, mask=m)
        _, _, o2, l2 = run_gpu(b)
        assert_close(bf16_tensor_to_f64(o1), l1.cpu().numpy().astype(np.float64),
                     bf16_tensor_to_f64(o2), l2.cpu().numpy().astype(np.float64),
                     "mask vs causal flag")


def test_decode_rows_even_position_mask():
    """Decode rows with a 2-D mask that keeps the even key positions."""
    b = W.make_batch([700, 2000, 31, 4096, 129], [1] * 5, 32, 8, 128, 16, seed=85)
    kv = int(-(-int(b.kv_lens.max()) // 16) * 16)
    m = np.zeros((b.batch, kv), bool)
    m[:, ::2] = True
    parity(b, mask=m, what="even positions")


def test_fully_masked_rows():
    b = W.make_batch([10, 200], [150, 1], 8, 2, 128, 16, seed=86)
    m = W.random_mask(b, "4d_heads", seed=87, keep=0.7)
    m[0, :, 5:40, :] = False   # rows 5..39 of sequence 0: nothing visible
    m[1, 3, :, :] = False      # head 3 of the decode row
    parity(b, mask=m, what="fully masked rows")


def test_unaligned_mask_width():
    """A mask whose key extent is not a multiple of 16 (the binding pads it)."""
    b = W.make_batch([33, 0], [90, 40], 8, 2, 64, 16, seed=88)
    m = W.random_mask(b, "4d_bcast", seed=89)[..., :int(b.kv_lens.max())]
    assert m.shape[-1] % 16 != 0
    parity(b, causal=False, mask=m, what="unaligned mask")
