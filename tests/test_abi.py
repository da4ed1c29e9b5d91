"""The C ABI library (no GPU needed): it builds, loads, exports every entry
point include/pcp.h declares, and rejects bad arguments on the host before
touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "pcp.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pcp_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from paged_chunked_prefill_gb300 import build
    build.build()
    import paged_chunked_prefill_gb300 as pcp
    return pcp.lib()


def test_header_declares_the_path():
    names = declared_functions()
    for n in ("pcp_compute_out_cache_loc", "pcp_kv_append", "pcp_paged_extend_attn",
              "pcp_extend_workspace_size", "pcp_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(7):
        s = lib.pcp_status_string(code).decode()
        assert s.startswith("PCP_")
    assert lib.pcp_status_string(99).decode() == "PCP_ERR_UNKNOWN"
    assert lib.pcp_abi_version() == 5
    lib.pcp_last_cuda_error.restype = ctypes.c_char_p
    assert lib.pcp_last_cuda_error().decode() == "no error"


def test_workspace_size(lib):
    import paged_chunked_prefill_gb300 as pcp
    a = pcp.workspace_size(8, 4096, 32, 8, 128)
    b = pcp.workspace_size(8, 8192, 32, 8, 128)
    assert 0 < a < b and a % 256 == 0
    assert pcp.workspace_size(8, 4096, 32, 8, 96) == 0        # unsupported head_dim
    assert pcp.workspace_size(8, 4096, 30, 8, 128) == 0       # Hq % Hkv != 0
    assert pcp.workspace_size(0, 0, 4, 4, 64) > 0


def test_host_validation_without_device(lib):
    """Arguments the host can check are rejected before any CUDA call."""
    P = ctypes.c_void_p
    dummy = ctypes.c_int32(0)
    err = ctypes.cast(ctypes.pointer(dummy), P)
    one = P(0x1000)
    st = lib.pcp_paged_extend_attn(one, one, one, one, one, P(0), 1, 10, one, one, 4, 16, 30, 8, 128,
                                   0, 0.0, one, one, one, 1 << 20, err, P(0))
    assert st == 1   # INVALID_ARG: 30 % 8 != 0
    st = lib.pcp_paged_extend_attn(one, one, one, one, one, P(0), 1, 10, one, one, 4, 16, 8, 8, 96,
                                   0, 0.0, one, one, one, 1 << 20, err, P(0))
    assert st == 2   # UNSUPPORTED head_dim
    st = lib.pcp_paged_extend_attn(one, one, one, one, one, P(0), 1, 10, one, one, 4, 16, 8, 8, 128,
                                   -1, 0.0, one, one, one, 1 << 20, err, P(0))
    assert st == 1   # negative window
    st = lib.pcp_paged_extend_attn(one, one, one, one, one, P(0), 1, 10, one, one, 4, 16, 8, 8, 128,
                                   0, 0.0, one, one, one, 16, err, P(0))
    assert st == 4   # workspace too small
    # a host copy of qo_indptr that disagrees with total_q, or decreases
    for host in ([0, 4, 9], [0, 6, 4, 10]):
        h = (ctypes.c_int32 * len(host))(*host)
        st = lib.pcp_paged_extend_attn(one, one, one, one, one, ctypes.cast(h, P),
                                       len(host) - 1, 10, one, one, 4, 16, 8, 8, 128, 0, 0.0,
                                       one, one, one, 1 << 30, err, P(0))
        assert st == 1, host
    st = lib.pcp_kv_append(one, one, one, 5, 2, 128, one, one, 10, P(0), P(0))
    assert st == 1   # no error word
    st = lib.pcp_compute_out_cache_loc(one, one, one, one, 2, 10, 0, 4, one, err, P(0))
    assert st == 1   # page_size 0
    # causal flag and mask descriptor
    f = lib.pcp_paged_extend_attn_masked
    def masked(causal, window, mask, sb, sh, sq):
        return f(one, one, one, one, one, P(0), 1, 10, one, one, 4, 16, 8, 8, 128, window, 0.0,
                 causal, mask, sb, sh, sq, 4, 64, one, one, one, 1 << 30, err, P(0))
    assert masked(2, 0, P(0), 0, 0, 0) == 1          # causal must be 0 or 1
    assert masked(0, 8, P(0), 0, 0, 0) == 1          # a window needs causal attention
    assert masked(1, 0, P(0x1008), 64, 0, 0) == 1    # mask not 16-byte aligned
    assert masked(1, 0, one, 40, 0, 0) == 1          # stride not a multiple of 16
    assert masked(1, 0, one, 64, 0, -16) == 1        # negative stride
    # per-call options: each kernel's events come both or not at all
    from paged_chunked_prefill_gb300._binding import CallOptions
    lib.pcp_paged_extend_attn_ex.restype = ctypes.c_int
    def ex(opts):
        return lib.pcp_paged_extend_attn_ex(
            one, one, one, one, one, P(0), 1, 10, one, one, 4, 16, 8, 8, 128, 0,
            ctypes.c_float(0.0), 1, P(0), ctypes.c_int64(0), ctypes.c_int64(0),
            ctypes.c_int64(0), 0, 0, one, one, one, ctypes.c_size_t(1 << 30), err, P(0),
            ctypes.byref(opts) if opts is not None else P(0))
    assert ex(CallOptions(one, P(0), P(0), P(0), 0)) == 1
    assert ex(CallOptions(P(0), P(0), P(0), one, 0)) == 1
    # the appended rows: k_new and v_new both or neither, 16-byte aligned;
    # out_cache_loc only with them
    none = P(0)
    assert ex(CallOptions(none, none, none, none, 0, none, one, none, none)) == 1
    assert ex(CallOptions(none, none, none, none, 0, none, none, one, none)) == 1
    assert ex(CallOptions(none, none, none, none, 0, none, P(0x1008), one, none)) == 1
    assert ex(CallOptions(none, none, none, none, 0, none, none, none, one)) == 1
    # the argument checks come before the options are looked at
    assert lib.pcp_paged_extend_attn_ex(
        one, one, one, one, one, P(0), 1, 10, one, one, 4, 16, 30, 8, 128, 0,
        ctypes.c_float(0.0), 1, P(0), ctypes.c_int64(0), ctypes.c_int64(0), ctypes.c_int64(0),
        0, 0, one, one, one, ctypes.c_size_t(1 << 30), err, P(0),
        ctypes.byref(CallOptions(one, P(0), P(0), P(0), 0))) == 1
    # the entry point without a workspace checks its arguments first, then
    # refuses calls larger than its fixed scratch (no device access either way)
    g = lib.pcp_paged_extend_attn_noalloc
    def noalloc(hq):
        return g(one, one, one, one, one, P(0), 4096, ctypes.c_int64(65536), one, one,
                 ctypes.c_int64(1), 16, hq, 8, 128, 0, ctypes.c_float(0.0), one, one, err, P(0))
    assert noalloc(32) == 4
    assert noalloc(30) == 1
    # empty work returns OK without touching the device
    assert lib.pcp_paged_extend_attn(P(0), P(0), P(0), P(0), P(0), P(0), 0, 0, P(0), P(0), 0, 16, 8,
                                     8, 128, 0, 0.0, P(0), P(0), P(0), 0, err, P(0)) == 0
    assert lib.pcp_kv_append(P(0), P(0), P(0), 0, 2, 128, P(0), P(0), 0, err, P(0)) == 0


def test_library_has_no_oracle_dependency():
    """The product package never imports the oracle."""
    pkg = os.path.join(ROOT, "paged_chunked_prefill_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in src.lower().replace("oracle-free", ""), f
