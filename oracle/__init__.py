"""FP64 CPU oracle for paged extend attention and KV append.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this package.  The
CUDA library never imports, links or calls it, and it shares no code with the
CUDA library.

The arithmetic lives in ``pcp_oracle.c`` (plain loops in double precision,
compiled with gcc, OpenMP over rows when available); this module only builds
it, loads it and marshals numpy arrays.  The header comment of
``pcp_oracle.c`` states the definition each function writes out and the
passages it follows.

Every function here is pinned by ``tests/test_oracle_pins.py``; none is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pcp_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK = 0
ERR_INVALID_ARG = 1
ERR_BAD_INDEX = 3


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"oracle {what} failed with code {code}")
        self.code = code


def build(force: bool = False) -> str:
    """Compile ``pcp_oracle.c`` into ``_build/liboracle.so`` (gcc, -O2, OpenMP
    when available).  Returns the library path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_out_cache_loc.argtypes = [i32, P, P, P, P, i32, i64, P]
        lib.oracle_kv_append.argtypes = [i64, i64, P, P, P, P, P, i64]
        lib.oracle_attention_rows.argtypes = [i32, P, P, P, P, P, P, P, i64, i32, i32, i32, i32,
                                              i32, dbl, i64, P, P, P, P]
        lib.oracle_attention.argtypes = [i32, P, P, P, P, P, P, P, i64, i32, i32, i32, i32, i32,
                                         dbl, P, P]
        mask_args = [i32, P, i64, i64, i64, i64, i64]
        lib.oracle_attention_rows_masked.argtypes = (
            [i32, P, P, P, P, P, P, P, i64, i32, i32, i32, i32, i32, dbl] + mask_args +
            [i64, P, P, P, P])
        lib.oracle_attention_masked.argtypes = (
            [i32, P, P, P, P, P, P, P, i64, i32, i32, i32, i32, i32, dbl] + mask_args + [P, P])
        for f in (lib.oracle_out_cache_loc, lib.oracle_kv_append, lib.oracle_attention_rows,
                  lib.oracle_attention, lib.oracle_attention_rows_masked,
                  lib.oracle_attention_masked, lib.oracle_num_threads, lib.oracle_version):
            f.restype = ctypes.c_int
        _lib = lib
        return lib


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _nonempty(a: np.ndarray, dtype) -> np.ndarray:
    a = _c(a, dtype)
    return a if a.size else np.zeros(1, dtype)


def num_threads() -> int:
    """Threads the oracle's parallel loop uses (OMP_NUM_THREADS, else all cores)."""
    return int(_load().oracle_num_threads())


def out_cache_loc(qo_indptr, kv_indptr, kv_indices, prefix_lens, page_size: int,
                  num_pages: int) -> np.ndarray:
    """Slots the new tokens of every sequence go to (int64 [total_q])."""
    lib = _load()
    qo = _c(qo_indptr, np.int32)
    kvp = _c(kv_indptr, np.int32)
    kvi = _nonempty(kv_indices, np.int32)
    pl = _nonempty(prefix_lens, np.int32)
    B = qo.shape[0] - 1
    out = np.zeros(max(int(qo[-1]), 1), dtype=np.int64)
    st = lib.oracle_out_cache_loc(B, _p(qo), _p(kvp), _p(kvi), _p(pl), int(page_size),
                                  int(num_pages), _p(out))
    if st != OK:
        raise OracleError(st, "out_cache_loc")
    return out[: int(qo[-1])]


def kv_append(k: np.ndarray, v: np.ndarray, loc: np.ndarray, k_pool: np.ndarray,
              v_pool: np.ndarray) -> None:
    """In place: k_pool[loc[t]] = k[t], v_pool[loc[t]] = v[t] (bf16 bit patterns)."""
    lib = _load()
    assert k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    assert k_pool.dtype == np.uint16 and v_pool.dtype == np.uint16
    n = int(np.asarray(k).shape[0])
    row = int(np.prod(k_pool.shape[1:]))
    k = _nonempty(k, np.uint16)
    v = _nonempty(v, np.uint16)
    loc = _nonempty(loc, np.int64)
    st = lib.oracle_kv_append(n, row, _p(k), _p(v), _p(loc), _p(k_pool), _p(v_pool),
                              k_pool.shape[0])
    if st != OK:
        raise OracleError(st, "kv_append")


def mask_view(mask, batch: int, n_q_heads: int):
    """A boolean mask as (uint8 array, b, h, q strides in elements, q extent,
    kv extent): 2-D [batch, kv] (one key mask per sequence) or 4-D
    [batch, 1 or Hq, 1 or q_len, kv]; size-1 head / query dimensions
    broadcast (stride 0)."""
    m = np.ascontiguousarray(np.asarray(mask, dtype=bool)).view(np.uint8)
    if m.ndim == 2:
        if m.shape[0] != batch:
            raise ValueError("mask batch mismatch")
        return m, m.shape[1], 0, 0, 1, m.shape[1]
    if m.ndim != 4 or m.shape[0] != batch or m.shape[1] not in (1, n_q_heads):
        raise ValueError("mask must be [B, kv] or [B, 1|Hq, 1|q, kv]")
    sb = m.shape[1] * m.shape[2] * m.shape[3]
    sh = 0 if m.shape[1] == 1 else m.shape[2] * m.shape[3]
    sq = 0 if m.shape[2] == 1 else m.shape[3]
    return m, sb, sh, sq, m.shape[2], m.shape[3]


def paged_extend_attn(q, qo_indptr, kv_indptr, kv_indices, prefix_lens, k_pool, v_pool,
                      page_size: int, n_q_heads: int, n_kv_heads: int, head_dim: int,
                      window: int = 0, sm_scale: float = 0.0,
                      rows: Optional[Tuple[np.ndarray, np.ndarray]] = None,
                      causal: bool = True, mask=None):
    """Extend attention in float64.

    Without ``rows``: returns out [total_q, Hq, D] and lse [total_q, Hq].
    With ``rows = (tokens, heads)``: returns out [n, D] and lse [n] for just
    those (row of q, query head) pairs.  ``causal=False`` lets every row see
    all of its sequence's keys; ``mask`` (see ``mask_view``) hides the keys
    whose entry is False.
    """
    lib = _load()
    qo = _c(qo_indptr, np.int32)
    kvp = _c(kv_indptr, np.int32)
    kvi = _nonempty(kv_indices, np.int32)
    pl = _nonempty(prefix_lens, np.int32)
    qb = _nonempty(q, np.uint16)
    kp = _c(k_pool, np.uint16)
    vp = _c(v_pool, np.uint16)
    B = qo.shape[0] - 1
    num_pages = kp.shape[0] // page_size
    args = (B, _p(qo), _p(kvp), _p(kvi), _p(pl), _p(qb), _p(kp), _p(vp), num_pages,
            int(page_size), int(n_q_heads), int(n_kv_heads), int(head_dim), int(window),
            float(sm_scale))
    if mask is None:
        m, margs = None, (int(bool(causal)), None, 0, 0, 0, 0, 0)
    else:
        m, sb, sh, sq, ql, kl = mask_view(mask, B, n_q_heads)
        margs = (int(bool(causal)), _p(m), sb, sh, sq, ql, kl)
    if rows is None:
        total_q = int(qo[-1])
        out = np.zeros((max(total_q, 1), n_q_heads, head_dim), dtype=np.float64)
        lse = np.zeros((max(total_q, 1), n_q_heads), dtype=np.float64)
        st = lib.oracle_attention_masked(*args, *margs, _p(out), _p(lse))
        if st != OK:
            raise OracleError(st, "attention")
        return out[:total_q], lse[:total_q]
    tok = _nonempty(rows[0], np.int64)
    head = _nonempty(rows[1], np.int32)
    n = int(np.asarray(rows[0]).shape[0])
    out = np.zeros((max(n, 1), head_dim), dtype=np.float64)
    lse = np.zeros(max(n, 1), dtype=np.float64)
    st = lib.oracle_attention_rows_masked(*args, *margs, n, _p(tok), _p(head), _p(out),
                                          _p(lse))
    if st != OK:
        raise OracleError(st, "attention_rows")
    return out[:n], lse[:n]


def run_batch(batch, rows=None, causal=True, mask=None):
    """Append a workload's chunk into copies of its pools, then attend.

    Returns (out_cache_loc, k_pool_after, v_pool_after, out, lse)."""
    loc = out_cache_loc(batch.qo_indptr, batch.kv_indptr, batch.kv_indices, batch.prefix_lens,
                        batch.page_size, batch.num_pages)
    kp = batch.k_pool.copy()
    vp = batch.v_pool.copy()
    kv_append(batch.k_new, batch.v_new, loc, kp, vp)
    out, lse = paged_extend_attn(batch.q, batch.qo_indptr, batch.kv_indptr, batch.kv_indices,
                                 batch.prefix_lens, kp, vp, batch.page_size, batch.n_q_heads,
                                 batch.n_kv_heads, batch.head_dim, batch.window,
                                 batch.sm_scale, rows=rows, causal=causal, mask=mask)
    return loc, kp, vp, out, lse
