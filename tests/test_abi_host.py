"""The C ABI without a GPU: the library loads, exports every function that
include/muon.h declares, and validates arguments on a host-only handle
(device = -1) before anything could be launched."""
import ctypes
import os
import re

import pytest

from muon_newton_schulz_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "muon.h")


@pytest.fixture(scope="module")
def lib():
    return B.load_library(build_if_missing=True)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(muon_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_function(lib):
    names = declared_functions()
    assert "muon_step" in names and "muon_create" in names
    for name in names:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert B.muon_status_string(B.MUON_OK) == "MUON_OK"
    assert B.muon_status_string(B.MUON_ERR_TIMEOUT) == "MUON_ERR_TIMEOUT"


def test_config_defaults(lib):
    c = B.muon_config_default()
    assert abs(c.beta - 0.95) < 1e-7 and c.ns_iters == 5 and c.mode == B.MUON_MODE_BF16
    assert (round(c.a, 4), round(c.b, 4), round(c.c, 4)) == (3.4445, -4.775, 2.0315)
    assert abs(c.scale_coeff - 0.2) < 1e-7 and abs(c.eps - 1e-7) < 1e-12
    assert c.nesterov == 0 and c.dampening == 0


def test_struct_layout_matches_header(lib):
    # 2 x int64, then pointer/int32/int32/int64, ... as declared
    assert ctypes.sizeof(B.muon_matrix_desc) == 8 * 2 + 8 + 4 + 4 + 8 + 8 * 2 + 8 * 2 + 4 + 4 + 8 * 2
    assert ctypes.sizeof(B.muon_config) == 10 * 4


@pytest.fixture()
def host_handle(lib):
    st, h = B.muon_create(None, -1)
    assert st == B.MUON_OK
    yield h
    B.muon_destroy(h)


def _desc(rows=256, cols=512, base=1 << 20, w_dtype=B.MUON_BF16, **kw):
    d = dict(rows=rows, cols=cols, W=base, w_dtype=w_dtype, ldw=cols,
             G=base + (1 << 24), ldg=cols, M=base + (2 << 24), ldm=cols, lr=2e-4)
    d.update(kw)
    return d


def _ws(h, items):
    arr, n = B.make_descs(items)
    return B.muon_workspace_size(h, arr, n)


def test_workspace_size_valid(host_handle):
    st, nbytes = _ws(host_handle, [_desc()])
    assert st == B.MUON_OK
    # X ping-pong as bf16 (hi, lo) pairs, A and B (bf16), plus small headers
    m, n = 256, 512
    body = 2 * m * n * 2 + 2 * m * n * 2 + 2 * m * m * 2
    assert body <= nbytes <= body + 64 * 1024


def test_workspace_tall_equals_wide(host_handle):
    st1, a = _ws(host_handle, [_desc(rows=256, cols=512)])
    st2, b = _ws(host_handle, [_desc(rows=512, cols=256)])
    assert st1 == st2 == B.MUON_OK and a == b


def test_workspace_fp32_mode_larger(lib):
    cfg = B.muon_config_default()
    cfg.mode = B.MUON_MODE_FP32_VALIDATE
    st, h = B.muon_create(cfg, -1)
    assert st == B.MUON_OK
    st, nbytes = _ws(h, [_desc()])
    assert st == B.MUON_OK
    m, n = 256, 512
    assert nbytes >= 2 * m * n * 4 + 2 * m * m * 4
    B.muon_destroy(h)


def test_empty_batch_and_empty_matrices(host_handle):
    arr, _ = B.make_descs([])
    assert B.muon_workspace_size(host_handle, arr, 0) == (B.MUON_OK, 0)
    st, nbytes = _ws(host_handle, [dict(rows=0, cols=7), dict(rows=5, cols=0)])
    assert st == B.MUON_OK and nbytes == 0
    arr, n = B.make_descs([dict(rows=0, cols=7)])
    assert B.muon_step(host_handle, arr, n, 0, 0, 0) == B.MUON_OK


@pytest.mark.parametrize("bad, why", [
    (dict(W=None), "NULL W"),
    (dict(G=None), "NULL G"),
    (dict(M=None), "NULL M"),
    (dict(rows=-1), "negative rows"),
    (dict(ldg=100), "ld < cols"),
    (dict(ldw=516), "ld not 16-byte multiple for bf16"),
    (dict(ldm=514), "ld not 16-byte multiple for fp32"),
    (dict(W=(1 << 20) + 8), "misaligned W"),
    (dict(G=(1 << 20) + 4096), "G overlaps W"),
    (dict(w_dtype=7), "bad dtype"),
    (dict(lr=float("nan")), "nan lr"),
    (dict(rows=40000, cols=40000), "too large"),
])
def test_invalid_descriptors(host_handle, bad, why):
    d = _desc(**bad)
    st, _ = _ws(host_handle, [d])
    assert st == B.MUON_ERR_INVALID_ARG, why
    assert B.muon_last_error_message(host_handle)
    arr, n = B.make_descs([d])
    assert B.muon_step(host_handle, arr, n, 1 << 30, 1 << 30, 0) == B.MUON_ERR_INVALID_ARG


def test_overlap_across_descriptors(host_handle):
    a = _desc(base=1 << 20)
    b = _desc(base=(1 << 20) + 128)  # b.W inside a.W
    st, _ = _ws(host_handle, [a, b])
    assert st == B.MUON_ERR_INVALID_ARG
    assert "overlap" in B.muon_last_error_message(host_handle)


def test_step_on_host_handle_is_unsupported_after_validation(host_handle):
    arr, n = B.make_descs([_desc()])
    assert B.muon_step(host_handle, arr, n, 1 << 30, 1 << 30, 0) == B.MUON_ERR_UNSUPPORTED


def test_negative_n(host_handle):
    arr, _ = B.make_descs([_desc()])
    assert B.muon_workspace_size(host_handle, arr, -1)[0] == B.MUON_ERR_INVALID_ARG


@pytest.mark.parametrize("field, value, status", [
    ("ns_iters", 65, B.MUON_ERR_INVALID_ARG),
    ("ns_iters", -1, B.MUON_ERR_INVALID_ARG),
    ("mode", 7, B.MUON_ERR_UNSUPPORTED),
    ("nesterov", 2, B.MUON_ERR_INVALID_ARG),
    ("dampening", -1, B.MUON_ERR_INVALID_ARG),
    ("eps", -1.0, B.MUON_ERR_INVALID_ARG),
    ("beta", float("inf"), B.MUON_ERR_INVALID_ARG),
])
def test_invalid_config(lib, field, value, status):
    cfg = B.muon_config_default()
    setattr(cfg, field, value)
    st, h = B.muon_create(cfg, -1)
    assert st == status


def test_create_without_gpu_is_unsupported(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st, h = B.muon_create(None, 0)
    assert st == B.MUON_ERR_UNSUPPORTED


def test_profiling_calls_on_host_handle(host_handle):
    assert B.muon_set_profiling(host_handle, True) == B.MUON_ERR_UNSUPPORTED
    assert B.muon_launch_count(host_handle) == 0


def test_workspace_overlapping_a_buffer_is_rejected(host_handle):
    base = 1 << 30
    d = _desc(base=base)
    arr, n = B.make_descs([d])
    st, need = B.muon_workspace_size(host_handle, arr, n)
    assert st == B.MUON_OK
    # a workspace that starts inside M (M is at base + 2^25)
    ws = base + (2 << 24) + 4096
    assert B.muon_step(host_handle, arr, n, ws, need, 0) == B.MUON_ERR_INVALID_ARG
    assert "workspace overlaps desc 0 M" in B.muon_last_error_message(host_handle)
    # one that ends inside W
    ws = base - need + 256
    ws -= ws % 256
    assert B.muon_step(host_handle, arr, n, ws, need, 0) == B.MUON_ERR_INVALID_ARG
    assert "workspace overlaps desc 0 W" in B.muon_last_error_message(host_handle)
    # one that ends right where W starts, and a disjoint one, pass validation
    # (and the host-only handle then refuses to run)
    assert B.muon_step(host_handle, arr, n, base - need, need, 0) == B.MUON_ERR_UNSUPPORTED
    assert B.muon_step(host_handle, arr, n, 1 << 34, need, 0) == B.MUON_ERR_UNSUPPORTED


def test_plan_counter_on_host_handle(host_handle):
    # a host-only handle validates but never builds a launch plan
    arr, n = B.make_descs([_desc()])
    B.muon_step(host_handle, arr, n, 1 << 32, 1 << 30, 0)
    assert B.muon_plan_builds(host_handle) == 0


def test_host_pipeline_workspace(host_handle):
    items = [_desc(base=(1 << 30) + k * (1 << 27)) for k in range(5)]
    arr, n = B.make_descs(items)
    st, one = B.muon_workspace_size(host_handle, arr, 1)
    assert st == B.MUON_OK
    sizes = {}
    for slots in (2, 3, 4):
        pl = B.make_pipeline(B.MUON_HOST_W | B.MUON_HOST_G | B.MUON_HOST_M, 1, slots)
        st, sizes[slots] = B.muon_host_workspace_size(host_handle, arr, n, pl)
        assert st == B.MUON_OK
    # one slot per chunk in flight: the step's workspace plus the staged W, G, M
    slot = sizes[2] // 2
    assert sizes[3] == 3 * slot and sizes[4] == 4 * slot
    staged = 256 * 512 * (2 + 4 + 4)
    assert one + staged <= slot <= one + staged + 4096
    # no more slots than chunks
    pl = B.make_pipeline(B.MUON_HOST_G, 5, 4)
    st, b = B.muon_host_workspace_size(host_handle, arr, n, pl)
    assert st == B.MUON_OK and b % 1024 == 0 and b >= 5 * 256 * 512 * 4


@pytest.mark.parametrize("host, chunk, slots, reserved", [(16, 1, 2, 0), (7, 0, 2, 0), (7, 1, 1, 0), (7, 1, 65, 0),
                                                          (7, 1, 2, 1)])
def test_host_pipeline_invalid(host_handle, host, chunk, slots, reserved):
    arr, n = B.make_descs([_desc()])
    pl = B.make_pipeline(host, chunk, slots)
    pl.reserved = reserved
    assert B.muon_host_workspace_size(host_handle, arr, n, pl)[0] == B.MUON_ERR_INVALID_ARG
    assert B.muon_step_host(host_handle, arr, n, pl, 1 << 34, 1 << 30, 0) == B.MUON_ERR_INVALID_ARG


def test_host_step_on_host_handle_is_unsupported(host_handle):
    arr, n = B.make_descs([_desc()])
    pl = B.make_pipeline(B.MUON_HOST_G, 1, 2)
    st, need = B.muon_host_workspace_size(host_handle, arr, n, pl)
    assert B.muon_step_host(host_handle, arr, n, pl, 1 << 34, need, 0) == B.MUON_ERR_UNSUPPORTED
    assert B.muon_step_host(host_handle, arr, n, pl, 1 << 34, need - 256, 0) == B.MUON_ERR_WORKSPACE
