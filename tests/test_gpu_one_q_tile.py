"""One-Q-tile items of the tensor-core kernel.

An item holds two Q tiles of one (sequence, KV head) unless the chunk's last
item has at most 128 / G positions left; such an item runs on one softmax
warpgroup, over 1 to 25 KV tiles here.  Decode-shaped chunks beside them may
join the tensor-core queue as one-Q-tile items too.  With the host copy of
qo_indptr a causal unmasked call with such items takes the instantiation in
which they alternate S/P buffers 0 and 1 over their KV tiles (odd and even
tile counts here); without it, or with a mask, the one in which each KV tile
runs QK^T, softmax and PV in turn.  Every row is compared
with the FP64 oracle, with and without the host copy of qo_indptr, on both
head sizes, windows, a boolean mask and page sizes that take TMA page boxes
and the cp.async gathers.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from helpers import assert_close, bf16_tensor_to_f64, run_gpu

pytestmark = pytest.mark.gpu


def _batch(D, page_size, window, seed):
    # G = 4 (16 / 4 heads), 32 positions per Q tile, 64 per item: chunks of
    # 20, 90 (64 + 26) and 160 (128 + 32) end in a one-Q-tile item; 97 (64 +
    # 33) does not.  Prefixes give 1 to 25 KV tiles, odd and even.
    P = [0, 130, 257, 1000, 2500, 3071, 77, 640]
    C = [20, 90, 160, 97, 20, 90, 4, 1]
    return W.make_batch(P, C, 16, 4, D, page_size, seed=seed, window=window,
                        name=f"one-Q-tile items, D={D}, ps={page_size}, window={window}")


def _check(b, host_hint, mask=None):
    """Every row against the oracle; rows that see no key give out = 0 and
    lse = -inf exactly."""
    _, _, out, lse = run_gpu(b, host_hint=host_hint, mask=mask)
    _, _, _, out_ref, lse_ref = oracle.run_batch(b, mask=mask)
    o = bf16_tensor_to_f64(out)
    l = lse.cpu().numpy().astype(np.float64)
    empty = np.isneginf(lse_ref)
    assert (np.isneginf(l) == empty).all()
    assert (o[empty] == 0).all()
    assert_close(o, np.where(empty, 0.0, l), out_ref, np.where(empty, 0.0, lse_ref),
                 f"{b.name}, host copy {host_hint}")


@pytest.mark.parametrize("host_hint", [True, False])
@pytest.mark.parametrize("D,page_size,window", [(128, 16, 0), (128, 16, 700), (64, 64, 0),
                                                (64, 1, 300), (128, 3, 0)])
def test_one_q_tile_items(D, page_size, window, host_hint):
    _check(_batch(D, page_size, window, seed=40 + D + page_size + window), host_hint)


@pytest.mark.parametrize("host_hint", [True, False])
def test_one_q_tile_items_with_a_mask(host_hint):
    b = _batch(128, 16, 0, seed=77)
    mask = W.random_mask(b, "2d", seed=78, keep=0.7)
    _check(b, host_hint, mask=mask)
