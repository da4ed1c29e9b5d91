"""ctypes binding of libpcp.so: argument marshalling only."""
from __future__ import annotations

import ctypes
import enum
import os
import threading
from typing import Optional, Tuple

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libpcp.so"
_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return os.path.join(_PKG, _LIB_NAME)


class Status(enum.IntEnum):
    OK = 0
    INVALID_ARG = 1
    UNSUPPORTED = 2
    BAD_INDEX = 3
    WORKSPACE = 4
    CUDA = 5
    TIMEOUT = 6


class CallOptions(ctypes.Structure):
    """``pcp_call_options``: per-call events around the tensor-core and row
    kernels, the stall that tests the kernels' timeout path, the host copy of
    prefix_lens, and the step's new K/V rows to append before attending."""
    _fields_ = [("tc_event_before", ctypes.c_void_p), ("tc_event_after", ctypes.c_void_p),
                ("rows_event_before", ctypes.c_void_p), ("rows_event_after", ctypes.c_void_p),
                ("test_stall_ns", ctypes.c_uint64), ("prefix_lens_host", ctypes.c_void_p),
                ("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p),
                ("out_cache_loc", ctypes.c_void_p)]


class PCPError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        msg = lib().pcp_status_string(int(status)).decode()
        if self.status == Status.CUDA:
            msg += f" ({lib().pcp_last_cuda_error().decode()})"
        super().__init__(f"{where}: {msg}")


def lib():
    """The loaded library.  Raises if libpcp.so has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise ImportError(
                f"{path} is missing: build it with `python -m paged_chunked_prefill_gb300.build` "
                "(there is no fallback implementation)")
        L = ctypes.CDLL(path)
        P, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                                ctypes.c_size_t)
        L.pcp_status_string.argtypes = [i32]
        L.pcp_status_string.restype = ctypes.c_char_p
        L.pcp_abi_version.argtypes = []
        L.pcp_abi_version.restype = i32
        L.pcp_last_cuda_error.argtypes = []
        L.pcp_last_cuda_error.restype = ctypes.c_char_p
        L.pcp_compute_out_cache_loc.argtypes = [P, P, P, P, i32, i64, i32, i64, P, P, P]
        L.pcp_compute_out_cache_loc.restype = i32
        L.pcp_kv_append.argtypes = [P, P, P, i64, i32, i32, P, P, i64, P, P]
        L.pcp_kv_append.restype = i32
        L.pcp_kv_append_paged.argtypes = [P, P, P, P, i32, i64, i32, i64, P, P, i32, i32, P, P,
                                          P, P, P]
        L.pcp_kv_append_paged.restype = i32
        L.pcp_extend_workspace_size.argtypes = [i32, i64, i32, i32, i32]
        L.pcp_extend_workspace_size.restype = sz
        L.pcp_paged_extend_attn.argtypes = [P, P, P, P, P, P, i32, i64, P, P, i64, i32, i32,
                                            i32, i32, i32, f32, P, P, P, sz, P, P]
        L.pcp_paged_extend_attn.restype = i32
        L.pcp_paged_extend_attn_masked.argtypes = [P, P, P, P, P, P, i32, i64, P, P, i64, i32,
                                                   i32, i32, i32, i32, f32, i32, P, i64, i64,
                                                   i64, i32, i32, P, P, P, sz, P, P]
        L.pcp_paged_extend_attn_masked.restype = i32
        L.pcp_paged_extend_attn_ex.argtypes = [P, P, P, P, P, P, i32, i64, P, P, i64, i32,
                                               i32, i32, i32, i32, f32, i32, P, i64, i64, i64,
                                               i32, i32, P, P, P, sz, P, P,
                                               ctypes.POINTER(CallOptions)]
        L.pcp_paged_extend_attn_ex.restype = i32
        L.pcp_pager_create.argtypes = [i64, i32]
        L.pcp_pager_create.restype = P
        L.pcp_pager_destroy.argtypes = [P]
        L.pcp_pager_destroy.restype = None
        L.pcp_pager_num_free.argtypes = [P]
        L.pcp_pager_num_free.restype = i64
        L.pcp_pager_num_held.argtypes = [P]
        L.pcp_pager_num_held.restype = i64
        L.pcp_pager_request_pages.argtypes = [P, i64, P, i64]
        L.pcp_pager_request_pages.restype = i64
        L.pcp_pager_release.argtypes = [P, i64]
        L.pcp_pager_release.restype = i32
        L.pcp_schedule_step.argtypes = [P, i32, P, P, P, i32, i32, P, P, P, P, P, P, i64, P,
                                        P, P, P, P]
        L.pcp_schedule_step.restype = i32
        L.pcp_pager_share.argtypes = [P, i64, i64, i64]
        L.pcp_pager_share.restype = i32
        L.pcp_pager_cache_prompt.argtypes = [P, i64, P, i64]
        L.pcp_pager_cache_prompt.restype = i64
        L.pcp_pager_match_prefix.argtypes = [P, i64, P, i64, P]
        L.pcp_pager_match_prefix.restype = i32
        L.pcp_pager_clear_cache.argtypes = [P]
        L.pcp_pager_clear_cache.restype = i32
        L.pcp_copy_page_slots.argtypes = [P, P, i64, i32, i32, i32, P, P, P, i32, P, P]
        L.pcp_copy_page_slots.restype = i32
        L.pcp_read_error.argtypes = [P, P, P]
        L.pcp_read_error.restype = i32
        _lib = L
        return L


def _check(status: int, where: str) -> None:
    if status != Status.OK:
        raise PCPError(status, where)


def _ptr(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _host_i32(a, n: int, name: str):
    """(pointer, owner) of an optional host int32 array of n entries."""
    if a is None:
        return ctypes.c_void_p(0), None
    if isinstance(a, torch.Tensor):
        if a.device.type != "cpu":
            raise ValueError(f"{name} must be a host (CPU) array")
        a = a.numpy()
    a = np.ascontiguousarray(a, dtype=np.int32)
    if a.ndim != 1 or a.shape[0] != n:
        raise ValueError(f"{name} must hold {n} int32 entries")
    return ctypes.c_void_p(a.ctypes.data), a


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t: torch.Tensor, name: str, dtype, device) -> None:
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


_err_bufs = {}
_ws_bufs = {}


def _dev_err(device: torch.device) -> torch.Tensor:
    key = (device.type, device.index)
    t = _err_bufs.get(key)
    if t is None:
        t = torch.zeros(1, dtype=torch.int32, device=device)
        _err_bufs[key] = t
    return t


def _workspace(device: torch.device, nbytes: int) -> torch.Tensor:
    key = (device.type, device.index)
    t = _ws_bufs.get(key)
    if t is None or t.numel() < nbytes:
        t = torch.empty(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
        _ws_bufs[key] = t
    return t


def read_error(dev_err: torch.Tensor) -> int:
    """Synchronise the current stream and return the device error word."""
    host = ctypes.c_int32(0)
    _check(lib().pcp_read_error(_ptr(dev_err), _stream(dev_err.device), ctypes.byref(host)),
           "pcp_read_error")
    return int(host.value)


def _finish(dev_err: torch.Tensor, own: bool, check: bool, where: str) -> None:
    if own and check:
        code = read_error(dev_err)
        if code != 0:
            dev_err.zero_()
            raise PCPError(code, where + " (device)")


def workspace_size(batch: int, total_q: int, n_q_heads: int, n_kv_heads: int,
                   head_dim: int) -> int:
    return int(lib().pcp_extend_workspace_size(batch, total_q, n_q_heads, n_kv_heads, head_dim))


def compute_out_cache_loc(qo_indptr: torch.Tensor, kv_indptr: torch.Tensor,
                          kv_indices: torch.Tensor, prefix_lens: torch.Tensor, page_size: int,
                          num_pages: int, total_q: Optional[int] = None,
                          out: Optional[torch.Tensor] = None,
                          dev_err: Optional[torch.Tensor] = None,
                          check: bool = True) -> torch.Tensor:
    """Slots (int64 [total_q]) where each new token of every chunk goes."""
    dev = qo_indptr.device
    for n, t in (("qo_indptr", qo_indptr), ("kv_indptr", kv_indptr),
                 ("kv_indices", kv_indices), ("prefix_lens", prefix_lens)):
        _need(t, n, torch.int32, dev)
    batch = qo_indptr.numel() - 1
    if total_q is None:
        total_q = int(qo_indptr[-1].item()) if batch > 0 else 0
    if out is None:
        out = torch.empty(total_q, dtype=torch.int64, device=dev)
    own = dev_err is None
    if own:
        dev_err = _dev_err(dev)
    _check(lib().pcp_compute_out_cache_loc(_ptr(qo_indptr), _ptr(kv_indptr), _ptr(kv_indices),
                                           _ptr(prefix_lens), batch, total_q, page_size,
                                           num_pages, _ptr(out), _ptr(dev_err), _stream(dev)),
           "pcp_compute_out_cache_loc")
    _finish(dev_err, own, check, "pcp_compute_out_cache_loc")
    return out


def kv_append(k: torch.Tensor, v: torch.Tensor, out_cache_loc: torch.Tensor,
              k_pool: torch.Tensor, v_pool: torch.Tensor,
              dev_err: Optional[torch.Tensor] = None, check: bool = True) -> None:
    """k_pool[out_cache_loc[t]] = k[t]; v_pool[...] = v[t]  (in place)."""
    dev = k.device
    for n, t in (("k", k), ("v", v), ("k_pool", k_pool), ("v_pool", v_pool)):
        _need(t, n, torch.bfloat16, dev)
    _need(out_cache_loc, "out_cache_loc", torch.int64, dev)
    if k.dim() != 3 or v.shape != k.shape or k_pool.shape != v_pool.shape:
        raise ValueError("k, v must be [n, Hkv, D] and the pools [slots, Hkv, D]")
    if tuple(k_pool.shape[1:]) != tuple(k.shape[1:]):
        raise ValueError("pool rows must match k rows")
    own = dev_err is None
    if own:
        dev_err = _dev_err(dev)
    _check(lib().pcp_kv_append(_ptr(k), _ptr(v), _ptr(out_cache_loc), k.shape[0], k.shape[1],
                               k.shape[2], _ptr(k_pool), _ptr(v_pool), k_pool.shape[0],
                               _ptr(dev_err), _stream(dev)), "pcp_kv_append")
    _finish(dev_err, own, check, "pcp_kv_append")


def kv_append_paged(qo_indptr: torch.Tensor, kv_indptr: torch.Tensor,
                    kv_indices: torch.Tensor, prefix_lens: torch.Tensor, page_size: int,
                    k: torch.Tensor, v: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                    out_cache_loc: Optional[torch.Tensor] = None,
                    dev_err: Optional[torch.Tensor] = None, check: bool = True) -> None:
    """Slot mapping and KV append in one kernel: each new token's slot from
    the page table, then k_pool[slot] = k[t], v_pool[slot] = v[t] (in place).
    out_cache_loc (int64 [total_q], optional) receives the slots."""
    dev = k.device
    for n, t in (("k", k), ("v", v), ("k_pool", k_pool), ("v_pool", v_pool)):
        _need(t, n, torch.bfloat16, dev)
    for n, t in (("qo_indptr", qo_indptr), ("kv_indptr", kv_indptr),
                 ("kv_indices", kv_indices), ("prefix_lens", prefix_lens)):
        _need(t, n, torch.int32, dev)
    if out_cache_loc is not None:
        _need(out_cache_loc, "out_cache_loc", torch.int64, dev)
    if k.dim() != 3 or v.shape != k.shape or k_pool.shape != v_pool.shape:
        raise ValueError("k, v must be [n, Hkv, D] and the pools [slots, Hkv, D]")
    if tuple(k_pool.shape[1:]) != tuple(k.shape[1:]) or k_pool.shape[0] % page_size:
        raise ValueError("pool rows must match k rows and hold whole pages")
    own = dev_err is None
    if own:
        dev_err = _dev_err(dev)
    _check(lib().pcp_kv_append_paged(_ptr(qo_indptr), _ptr(kv_indptr), _ptr(kv_indices),
                                     _ptr(prefix_lens), qo_indptr.numel() - 1, k.shape[0],
                                     page_size, k_pool.shape[0] // page_size, _ptr(k), _ptr(v),
                                     k.shape[1], k.shape[2], _ptr(k_pool), _ptr(v_pool),
                                     _ptr(out_cache_loc), _ptr(dev_err), _stream(dev)),
           "pcp_kv_append_paged")
    _finish(dev_err, own, check, "pcp_kv_append_paged")


def _mask_args(mask: Optional[torch.Tensor], batch: int, n_q_heads: int, device):
    """(tensor kept alive, pointer, b/h/q strides, q extent, kv extent) of a
    boolean mask: 2-D [batch, kv] or 4-D [batch, 1|Hq, 1|q, kv].  A mask whose
    rows are not 16-byte aligned is copied into a padded one."""
    if mask is None:
        return None, ctypes.c_void_p(0), 0, 0, 0, 0, 0
    if mask.dtype != torch.bool or mask.device != device:
        raise TypeError(f"mask must be a bool tensor on {device}")
    if mask.dim() == 2:
        mask = mask.view(mask.shape[0], 1, 1, mask.shape[1])
    if mask.dim() != 4 or mask.shape[0] != batch or mask.shape[1] not in (1, n_q_heads):
        raise ValueError("mask must be [B, kv] or [B, 1|Hq, 1|q, kv]")
    kv = mask.shape[3]
    if kv % 16 != 0 or not mask.is_contiguous() or mask.data_ptr() % 16 != 0:
        padded = torch.zeros(mask.shape[:3] + (-(-kv // 16) * 16,), dtype=torch.bool,
                             device=device)
        padded[..., :kv] = mask
        mask = padded
    sq = 0 if mask.shape[2] == 1 else mask.stride(2)
    sh = 0 if mask.shape[1] == 1 else mask.stride(1)
    return (mask, ctypes.c_void_p(mask.data_ptr()), mask.stride(0), sh, sq, mask.shape[2], kv)


def paged_extend_attn(q: torch.Tensor, qo_indptr: torch.Tensor, kv_indptr: torch.Tensor,
                      kv_indices: torch.Tensor, prefix_lens: torch.Tensor,
                      k_pool: torch.Tensor, v_pool: torch.Tensor, page_size: int,
                      n_q_heads: int, n_kv_heads: int, head_dim: int, window: int = 0,
                      sm_scale: float = 0.0, *, out: Optional[torch.Tensor] = None,
                      lse: Optional[torch.Tensor] = None,
                      workspace: Optional[torch.Tensor] = None,
                      dev_err: Optional[torch.Tensor] = None,
                      qo_indptr_host=None, causal: bool = True,
                      mask: Optional[torch.Tensor] = None,
                      tc_events=None, rows_events=None, test_stall_ns: int = 0,
                      prefix_lens_host=None, k_new: Optional[torch.Tensor] = None,
                      v_new: Optional[torch.Tensor] = None,
                      out_cache_loc: Optional[torch.Tensor] = None,
                      check: bool = True) -> Tuple[torch.Tensor, torch.Tensor]:
    """Extend attention of every query row over its cached prefix and own
    chunk (bottom-right causal, GQA, optional window).  Returns (out, lse):
    out bf16 [total_q, Hq, D], lse float32 [total_q, Hq] (natural log).

    qo_indptr_host: optional host copy of qo_indptr (numpy int32 array or CPU
    int32 tensor); with it the call skips the launch of a kernel that would
    have no work.
    prefix_lens_host: optional host copy of prefix_lens; with qo_indptr_host
    the host decides whether the decode-shaped chunks of a call with
    tensor-core work join the tensor-core queue (otherwise the planner
    kernel decides it on the device), and skips the row kernel and the
    combine when they do.
    causal=False: every row sees all keys of its sequence (no window).
    mask: optional bool tensor (True = keep) of shape [B, kv] or
    [B, 1|Hq, 1|q, kv], indexed by the row inside the chunk and the key
    position, applied on top of the causal rule.
    tc_events / rows_events: optional (before, after) torch.cuda.Event pairs
    recorded around the tensor-core / row kernel of this call.
    test_stall_ns: 0, or the limit of a wait that nothing ends, made by every
    CTA of the kernels the call launches (a test of their timeout path: the
    call then reports PCP_ERR_TIMEOUT).
    k_new, v_new: optional bf16 [total_q, Hkv, D] new K/V rows of the step;
    the call first appends them into k_pool / v_pool (as kv_append_paged
    does, in the planner's launch) and then attends.  out_cache_loc (int64
    [total_q], optional, with k_new) receives the slots."""
    dev = q.device
    _need(q, "q", torch.bfloat16, dev)
    _need(k_pool, "k_pool", torch.bfloat16, dev)
    _need(v_pool, "v_pool", torch.bfloat16, dev)
    for n, t in (("qo_indptr", qo_indptr), ("kv_indptr", kv_indptr),
                 ("kv_indices", kv_indices), ("prefix_lens", prefix_lens)):
        _need(t, n, torch.int32, dev)
    if q.dim() != 3 or q.shape[1] != n_q_heads or q.shape[2] != head_dim:
        raise ValueError("q must be [total_q, n_q_heads, head_dim]")
    if k_pool.shape[0] % page_size != 0:
        raise ValueError("pool slots must be a multiple of page_size")
    batch = qo_indptr.numel() - 1
    total_q = q.shape[0]
    num_pages = k_pool.shape[0] // page_size
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(total_q, n_q_heads, dtype=torch.float32, device=dev)
    need = workspace_size(batch, total_q, n_q_heads, n_kv_heads, head_dim)
    if workspace is None:
        workspace = _workspace(dev, need)
    own = dev_err is None
    if own:
        dev_err = _dev_err(dev)
    host_ptr, host_keep = _host_i32(qo_indptr_host, batch + 1, "qo_indptr_host")
    pl_ptr, pl_keep = _host_i32(prefix_lens_host, batch, "prefix_lens_host")
    if (k_new is None) != (v_new is None):
        raise ValueError("k_new and v_new go together")
    if k_new is not None:
        _need(k_new, "k_new", torch.bfloat16, dev)
        _need(v_new, "v_new", torch.bfloat16, dev)
        if tuple(k_new.shape) != (total_q, n_kv_heads, head_dim) or v_new.shape != k_new.shape:
            raise ValueError("k_new, v_new must be [total_q, n_kv_heads, head_dim]")
    if out_cache_loc is not None:
        if k_new is None:
            raise ValueError("out_cache_loc comes with k_new / v_new")
        _need(out_cache_loc, "out_cache_loc", torch.int64, dev)
    if (tc_events is not None or rows_events is not None or test_stall_ns or
            prefix_lens_host is not None or k_new is not None):
        ev = lambda e: ctypes.c_void_p(e.cuda_event) if e is not None else ctypes.c_void_p(0)
        tb, ta = tc_events if tc_events is not None else (None, None)
        rb, ra = rows_events if rows_events is not None else (None, None)
        opts = CallOptions(ev(tb), ev(ta), ev(rb), ev(ra), int(test_stall_ns), pl_ptr,
                           _ptr(k_new), _ptr(v_new), _ptr(out_cache_loc))
        mkeep, mptr, sb, sh, sq, mq, mkv = _mask_args(mask, batch, n_q_heads, dev)
        _check(lib().pcp_paged_extend_attn_ex(
            _ptr(q), _ptr(qo_indptr), _ptr(kv_indptr), _ptr(kv_indices), _ptr(prefix_lens),
            host_ptr, batch, total_q, _ptr(k_pool), _ptr(v_pool), num_pages, page_size,
            n_q_heads, n_kv_heads, head_dim, window, float(sm_scale), int(bool(causal)), mptr,
            sb, sh, sq, mq, mkv, _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
            _ptr(dev_err), _stream(dev), ctypes.byref(opts)), "pcp_paged_extend_attn_ex")
        del mkeep
    elif causal and mask is None:
        _check(lib().pcp_paged_extend_attn(
            _ptr(q), _ptr(qo_indptr), _ptr(kv_indptr), _ptr(kv_indices), _ptr(prefix_lens),
            host_ptr, batch, total_q, _ptr(k_pool), _ptr(v_pool), num_pages, page_size,
            n_q_heads, n_kv_heads, head_dim, window, float(sm_scale), _ptr(out), _ptr(lse),
            _ptr(workspace), workspace.numel(), _ptr(dev_err), _stream(dev)),
            "pcp_paged_extend_attn")
    else:
        mkeep, mptr, sb, sh, sq, mq, mkv = _mask_args(mask, batch, n_q_heads, dev)
        _check(lib().pcp_paged_extend_attn_masked(
            _ptr(q), _ptr(qo_indptr), _ptr(kv_indptr), _ptr(kv_indices), _ptr(prefix_lens),
            host_ptr, batch, total_q, _ptr(k_pool), _ptr(v_pool), num_pages, page_size,
            n_q_heads, n_kv_heads, head_dim, window, float(sm_scale), int(bool(causal)), mptr,
            sb, sh, sq, mq, mkv, _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
            _ptr(dev_err), _stream(dev)), "pcp_paged_extend_attn_masked")
        del mkeep
    del host_keep, pl_keep
    _finish(dev_err, own, check, "pcp_paged_extend_attn")
    return out, lse


def copy_page_slots(k_pool: torch.Tensor, v_pool: torch.Tensor, page_size: int,
                    src_pages: torch.Tensor, dst_pages: torch.Tensor, n_slots: torch.Tensor,
                    dev_err: Optional[torch.Tensor] = None, check: bool = True) -> None:
    """Copy-on-write on the device: slots [0, n_slots[c]) of page
    src_pages[c] -> page dst_pages[c], K and V (int32 device tensors)."""
    dev = k_pool.device
    _need(k_pool, "k_pool", torch.bfloat16, dev)
    _need(v_pool, "v_pool", torch.bfloat16, dev)
    for n, t in (("src_pages", src_pages), ("dst_pages", dst_pages), ("n_slots", n_slots)):
        _need(t, n, torch.int32, dev)
    if k_pool.shape != v_pool.shape or k_pool.dim() != 3 or k_pool.shape[0] % page_size:
        raise ValueError("pools must be [num_pages * page_size, Hkv, D]")
    own = dev_err is None
    if own:
        dev_err = _dev_err(dev)
    _check(lib().pcp_copy_page_slots(_ptr(k_pool), _ptr(v_pool), k_pool.shape[0] // page_size,
                                     page_size, k_pool.shape[1], k_pool.shape[2],
                                     _ptr(src_pages), _ptr(dst_pages), _ptr(n_slots),
                                     src_pages.numel(), _ptr(dev_err), _stream(dev)),
           "pcp_copy_page_slots")
    _finish(dev_err, own, check, "pcp_copy_page_slots")


class Pager:
    """Host-side page pool and chunk planner (``pcp_pager_*``,
    ``pcp_schedule_step``): argument marshalling only."""

    def __init__(self, num_pages: int, page_size: int):
        self._h = lib().pcp_pager_create(int(num_pages), int(page_size))
        if not self._h:
            raise ValueError("pcp_pager_create: bad arguments")
        self.page_size = int(page_size)
        self._bufs = None
        self._nrows, self._ncp = ctypes.c_int32(0), ctypes.c_int32(0)
        self._nrows_ref, self._ncp_ref = ctypes.byref(self._nrows), ctypes.byref(self._ncp)

    def close(self) -> None:
        if self._h:
            lib().pcp_pager_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def num_free(self) -> int:
        return int(lib().pcp_pager_num_free(self._h))

    def request_pages(self, req_id: int) -> np.ndarray:
        n = int(lib().pcp_pager_request_pages(self._h, int(req_id), None, 0))
        out = np.zeros(max(n, 1), np.int32)
        lib().pcp_pager_request_pages(self._h, int(req_id), out.ctypes.data_as(ctypes.c_void_p),
                                      n)
        return out[:n]

    def release(self, req_id: int) -> None:
        _check(lib().pcp_pager_release(self._h, int(req_id)), "pcp_pager_release")

    def share(self, src_req: int, dst_req: int, n_tokens: int) -> None:
        """dst_req takes read-only references to src_req's pages holding its
        first n_tokens tokens."""
        _check(lib().pcp_pager_share(self._h, int(src_req), int(dst_req), int(n_tokens)),
               "pcp_pager_share")

    def cache_prompt(self, req_id: int, tokens) -> int:
        """Enter the request's full pages into the prefix index; returns the
        pages newly entered."""
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        n = int(lib().pcp_pager_cache_prompt(self._h, int(req_id),
                                             t.ctypes.data_as(ctypes.c_void_p), t.shape[0]))
        if n < 0:
            raise ValueError("pcp_pager_cache_prompt: bad arguments")
        return n

    def match_prefix(self, req_id: int, tokens) -> int:
        """Attach the longest cached run of whole pages matching the prompt
        (leaving at least its last token); returns the tokens covered."""
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        hit = ctypes.c_int64(0)
        _check(lib().pcp_pager_match_prefix(self._h, int(req_id),
                                            t.ctypes.data_as(ctypes.c_void_p), t.shape[0],
                                            ctypes.byref(hit)), "pcp_pager_match_prefix")
        return int(hit.value)

    def clear_cache(self) -> None:
        _check(lib().pcp_pager_clear_cache(self._h), "pcp_pager_clear_cache")

    def schedule_step(self, req_ids, total_lens, num_computed, budget: int,
                      state_block: int = 0) -> dict:
        """Plan one step; returns numpy arrays row_req, qo_indptr,
        prefix_lens, kv_indptr, kv_indices and sample (bool)."""
        ids = np.ascontiguousarray(req_ids, dtype=np.int64)
        tot = np.ascontiguousarray(total_lens, dtype=np.int32)
        comp = np.ascontiguousarray(num_computed, dtype=np.int32)
        n = int(ids.shape[0])
        if tot.shape != (n,) or comp.shape != (n,):
            raise ValueError("req_ids, total_lens and num_computed must have one entry each")
        L = lib()
        cap = int(L.pcp_pager_num_held(self._h)) + int(L.pcp_pager_num_free(self._h)) + 1
        # output buffers are kept between steps and grown when too small; the
        # results handed back are copies
        b = self._bufs
        if b is None or b["n"] < n + 1 or b["cap"] < cap:
            m = max(n + 1, 2 * b["n"] if b else 0)
            k = max(cap, 2 * b["cap"] if b else 0)
            b = self._bufs = {"n": m, "cap": k, "kvi": np.empty(k, np.int32),
                              "smp": np.empty(m, np.uint8),
                              **{x: np.empty(m, np.int32) for x in (
                                  "row_req", "qo", "pre", "kvp", "csrc", "cdst", "cslots")}}
        kvi = b["kvi"]
        _check(L.pcp_schedule_step(self._h, n, ids.ctypes.data, tot.ctypes.data,
                                   comp.ctypes.data, int(budget), int(state_block),
                                   self._nrows_ref, b["row_req"].ctypes.data, b["qo"].ctypes.data,
                                   b["pre"].ctypes.data, b["kvp"].ctypes.data, kvi.ctypes.data,
                                   int(b["cap"]), b["smp"].ctypes.data, self._ncp_ref,
                                   b["csrc"].ctypes.data, b["cdst"].ctypes.data,
                                   b["cslots"].ctypes.data),
               "pcp_schedule_step")
        r = int(self._nrows.value)
        c = int(self._ncp.value)
        kvp = b["kvp"]
        return {"row_req": b["row_req"][:r].copy(), "qo_indptr": b["qo"][:r + 1].copy(),
                "prefix_lens": b["pre"][:r].copy(), "kv_indptr": kvp[:r + 1].copy(),
                "kv_indices": kvi[:int(kvp[r])].copy(), "sample": b["smp"][:r].astype(bool),
                "copy_src": b["csrc"][:c].copy(), "copy_dst": b["cdst"][:c].copy(),
                "copy_slots": b["cslots"][:c].copy()}
