"""The C-ABI library: it loads, exports every symbol include/moe.h declares, and
its host-side validation rejects bad calls before touching the GPU (no CUDA call
is made on these paths, so they run on a machine without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def m():
    import __graft_entry__

    __graft_entry__.build()
    import mixture_experts_layer_index_gb300 as mod

    return mod


def _declared():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(m):
    names = _declared()
    assert len(names) >= 10
    lib = ctypes.CDLL(m.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(m.EXPORTED)


def test_status_strings(m):
    for s in range(7):
        assert m.moe_status_string(s) and m.moe_status_string(s) != "unknown status"
    assert m.moe_status_string(99) == "unknown status"


def test_workspace_size_and_path(m):
    p = m.problem(16, 8, 2, 256, 128)
    assert m.moe_select_path(p) == m.MOE_PATH_GROUPED
    assert m.moe_workspace_size(p) > 0
    q = m.problem(1, 192, 8, 4096, 192, "fp8_tensor")
    assert m.moe_select_path(q) == m.MOE_PATH_ROUTE_DIRECT
    # AUTO crossovers: per-tensor FP8 up to T = 96, blockwise up to T = 64, and T*k <= 1024
    assert m.moe_select_path(m.problem(96, 192, 8, 4096, 192, "fp8_tensor")) == m.MOE_PATH_ROUTE_DIRECT
    assert m.moe_select_path(m.problem(97, 192, 8, 4096, 192, "fp8_tensor")) == m.MOE_PATH_GROUPED
    assert m.moe_select_path(m.problem(96, 192, 16, 4096, 192, "fp8_tensor")) == m.MOE_PATH_GROUPED
    assert m.moe_select_path(m.problem(64, 128, 8, 2048, 768, "fp8_block")) == m.MOE_PATH_ROUTE_DIRECT
    assert m.moe_select_path(m.problem(65, 128, 8, 2048, 768, "fp8_block")) == m.MOE_PATH_GROUPED
    assert m.moe_select_path(m.problem(40, 128, 32, 2048, 768, "fp8_block")) == m.MOE_PATH_GROUPED
    assert m.moe_select_path(m.problem(10**6, 16, 8, 1024, 1024)) == m.MOE_PATH_GROUPED
    assert m.moe_workspace_size(q) > 0
    # unsupported / invalid problems have no workspace
    assert m.moe_workspace_size(m.problem(16, 600, 2, 256, 128)) == 0
    assert m.moe_workspace_size(m.problem(16, 8, 9, 256, 128)) == 0
    assert m.moe_workspace_size(m.problem(16, 8, 2, 250, 128)) == 0
    assert m.moe_workspace_size(m.problem(16, 8, 2, 256, 128, "bf16", m.MOE_PATH_ROUTE_DIRECT)) == 0
    assert m.moe_workspace_size(m.problem(200, 128, 8, 2048, 768, "fp8_block", m.MOE_PATH_ROUTE_DIRECT)) == 0
    assert m.moe_workspace_size(m.problem(1, 128, 8, 2048, 96, "fp8_block")) == 0
    # shapes the route-MMA page's dispatch admits: blockwise with a 64-column last scale
    # group of I, per-tensor with H % 128 == 64; the grouped path takes them
    assert m.moe_workspace_size(m.problem(1, 128, 8, 2048, 192, "fp8_block")) > 0
    assert m.moe_select_path(m.problem(1, 128, 8, 2048, 192, "fp8_block")) == m.MOE_PATH_ROUTE_DIRECT
    assert m.moe_select_path(m.problem(512, 128, 8, 2048, 192, "fp8_block")) == m.MOE_PATH_GROUPED
    assert m.moe_select_path(m.problem(1, 192, 8, 4032, 192, "fp8_tensor")) == m.MOE_PATH_ROUTE_DIRECT
    assert m.moe_workspace_size(m.problem(1, 192, 8, 4032, 192, "fp8_tensor", m.MOE_PATH_ROUTE_DIRECT)) > 0
    assert m.moe_workspace_size(m.problem(512, 192, 8, 4032, 192, "fp8_tensor")) > 0
    # grows with T
    a = m.moe_workspace_size(m.problem(1024, 16, 8, 1024, 1024))
    b = m.moe_workspace_size(m.problem(2048, 16, 8, 1024, 1024))
    assert b > a


FAKE = 1 << 20  # an aligned, never-dereferenced address: validation fails before any use


def _fwd(m, p, x=FAKE, s=FAKE, w1=FAKE, w2=FAKE, s1=None, s2=None, y=FAKE, ws=FAKE, nb=1 << 40):
    return m.raw_status("moe_forward", ctypes.byref(p), x, s, w1, w2, s1, s2, y, ws, nb, None)


def test_forward_validation_without_launch(m):
    p = m.problem(16, 8, 2, 256, 128)
    assert _fwd(m, p, x=None) == m.MOE_ERR_INVALID_ARG
    assert _fwd(m, p, y=None) == m.MOE_ERR_INVALID_ARG
    assert _fwd(m, p, x=FAKE + 2) == m.MOE_ERR_INVALID_ARG  # misaligned
    assert _fwd(m, p, s1=FAKE) == m.MOE_ERR_INVALID_ARG      # scales with bf16
    assert _fwd(m, p, ws=None) == m.MOE_ERR_WORKSPACE
    assert _fwd(m, p, nb=16) == m.MOE_ERR_WORKSPACE
    assert _fwd(m, m.problem(16, 8, 9, 256, 128)) == m.MOE_ERR_INVALID_ARG
    assert _fwd(m, m.problem(16, 8, 0, 256, 128)) == m.MOE_ERR_INVALID_ARG
    assert _fwd(m, m.problem(-1, 8, 2, 256, 128)) == m.MOE_ERR_INVALID_ARG
    assert _fwd(m, m.problem(16, 1000, 2, 256, 128)) == m.MOE_ERR_UNSUPPORTED
    assert _fwd(m, m.problem(16, 8, 2, 100, 128)) == m.MOE_ERR_UNSUPPORTED
    q = m.problem(2, 32, 8, 512, 192, "fp8_tensor")
    assert _fwd(m, q) == m.MOE_ERR_INVALID_ARG               # FP8 needs both scales
    assert _fwd(m, q, s1=FAKE) == m.MOE_ERR_INVALID_ARG
    assert _fwd(m, q, s1=FAKE, s2=FAKE + 1) == m.MOE_ERR_INVALID_ARG
    assert _fwd(m, q, s1=FAKE, s2=FAKE, nb=10) == m.MOE_ERR_WORKSPACE
    assert m.raw_status("moe_forward", None, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, FAKE, 1, None) == \
        m.MOE_ERR_INVALID_ARG
    # T == 0 is a valid empty call: nothing to do, nothing launched
    assert _fwd(m, m.problem(0, 8, 2, 256, 128), x=None, y=None, ws=None, nb=0) == m.MOE_OK


def test_route_shuffle_tilemap_validation_without_launch(m):
    assert m.raw_status("moe_route", FAKE, 4, 8, 9, FAKE, FAKE, None) == m.MOE_ERR_INVALID_ARG
    assert m.raw_status("moe_route", None, 4, 8, 2, FAKE, FAKE, None) == m.MOE_ERR_INVALID_ARG
    assert m.raw_status("moe_route", FAKE, 4, 600, 2, FAKE, FAKE, None) == m.MOE_ERR_UNSUPPORTED
    assert m.raw_status("moe_route", None, 0, 8, 2, None, None, None) == m.MOE_OK
    need = m.moe_shuffle_workspace_size(100, 16, 4)
    assert need > 0
    assert m.raw_status("moe_shuffle", FAKE, 100, 16, 4, FAKE, FAKE, FAKE, FAKE, FAKE, need - 1, None) == \
        m.MOE_ERR_WORKSPACE
    assert m.raw_status("moe_shuffle", FAKE, 100, 16, 4, FAKE, FAKE, FAKE, FAKE, None, need, None) == \
        m.MOE_ERR_WORKSPACE
    assert m.raw_status("moe_shuffle", None, 100, 16, 4, FAKE, FAKE, FAKE, FAKE, FAKE, need, None) == \
        m.MOE_ERR_INVALID_ARG
    assert m.raw_status("moe_tile_map", FAKE, 16, 0, FAKE, FAKE, 10, FAKE, 1 << 20, None) == m.MOE_ERR_INVALID_ARG
    assert m.raw_status("moe_tile_map", FAKE, 16, 128, FAKE + 4, FAKE, 10, FAKE, 1 << 20, None) == \
        m.MOE_ERR_INVALID_ARG
    assert m.raw_status("moe_tile_map", FAKE, 16, 128, FAKE, FAKE, 10, FAKE, 8, None) == m.MOE_ERR_WORKSPACE


def test_package_fails_loudly_without_library(tmp_path, monkeypatch, m):
    monkeypatch.setattr(m, "_lib", None)
    monkeypatch.setattr(m, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        m.moe_workspace_size(m.problem(16, 8, 2, 256, 128))
