"""The C-ABI library builds, loads and exports every entry point its headers
declare; host-side argument checks answer without touching a GPU."""

import ctypes
import glob
import os
import re

import pytest

from quantized_moe_transformer_gb300 import binding as qb
from quantized_moe_transformer_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return qb.lib()


def declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names.update(re.findall(r"\b(qmoe_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_entry_points():
    names = declared_symbols()
    for required in ("qmoe_moe_route", "qmoe_moe_forward", "qmoe_moe_workspace_bytes"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert set(qb.exported_symbols()) <= set(declared_symbols())


def test_status_strings(lib):
    assert lib.qmoe_status_str(0) == b"ok"
    assert b"workspace" in lib.qmoe_status_str(-4)
    assert lib.qmoe_status_str(12345) == b"unknown status"


def _desc(H=2048, E=256, k=8, F=512, shared=True, **kw):
    fake = ctypes.c_void_p(4096)          # never dereferenced by host checks
    d = qb.MoeDesc(H, E, k, F, 0, 1, fake, fake, fake, fake,
                   fake if shared else None, fake if shared else None, fake if shared else None)
    for key, v in kw.items():
        setattr(d, key, v)
    return d


def test_workspace_sizes_are_host_computed(lib):
    d = _desc()
    small = lib.qmoe_moe_workspace_bytes(ctypes.byref(d), 1)
    big = lib.qmoe_moe_workspace_bytes(ctypes.byref(d), 4096)
    assert 0 < small < big
    # y [T*k + T][H] fp32 alone at 4096 rows
    assert big >= (4096 * 8 + 4096) * 2048 * 4
    assert lib.qmoe_moe_workspace_bytes(ctypes.byref(d), 0) == 0
    lay = qb.MoeWsLayout()
    assert lib.qmoe_moe_workspace_layout(ctypes.byref(d), 16, ctypes.byref(lay)) == 0
    assert lay.ids % 256 == 0 and lay.y % 256 == 0 and lay.y > lay.perm > lay.offsets


@pytest.mark.parametrize("field,value", [("H", 300), ("F", 100), ("E", 0), ("E", 2000), ("k", 0),
                                         ("k", 17), ("gate_type", 7)])
def test_bad_descriptor_rejected(lib, field, value):
    d = _desc(**{field: value})
    r = lib.qmoe_moe_forward(ctypes.byref(d), None, None, None, None, None, 1, None, 0, None)
    assert r == -1
    assert lib.qmoe_moe_workspace_bytes(ctypes.byref(d), 1) == 0


def test_partial_shared_expert_rejected(lib):
    d = _desc()
    d.Su = None
    assert lib.qmoe_moe_forward(ctypes.byref(d), None, None, None, None, None, 1, None, 0, None) == -2


def test_misaligned_weights_rejected(lib):
    d = _desc()
    d.Wg = ctypes.c_void_p(4096 + 8)
    assert lib.qmoe_moe_forward(ctypes.byref(d), None, None, None, None, None, 1, None, 0, None) == -3


def test_null_buffers_rejected(lib):
    d = _desc()
    assert lib.qmoe_moe_forward(ctypes.byref(d), None, None, None, None, None, 4, None, 0, None) == -2
    # ids without w
    r = lib.qmoe_moe_forward(ctypes.byref(d), ctypes.c_void_p(4096), None, ctypes.c_void_p(4096), None,
                             ctypes.c_void_p(8192), 4, ctypes.c_void_p(1 << 20), 1 << 30, None)
    assert r == -2


def test_zero_rows_is_a_no_op(lib):
    d = _desc()
    assert lib.qmoe_moe_forward(ctypes.byref(d), None, None, None, None, None, 0, None, 0, None) == 0
    assert lib.qmoe_last_path() == 0


def test_route_argument_checks(lib):
    assert lib.qmoe_moe_route(None, None, 1, 2048, 256, 0, None, None, None, 0, None) == -1
    assert lib.qmoe_moe_route(None, None, 0, 2048, 256, 8, None, None, None, 0, None) == 0
    assert lib.qmoe_moe_route(None, None, 1, 2048, 256, 8, None, None, None, 0, None) == -2


def test_route_workspace_holds_router_parts(lib):
    """From 256 rows the router runs on the tensor cores: the workspace holds
    Wr's three bf16 parts and at least 4 slices of partial logits."""
    T, H, E = 4096, 2048, 256
    parts = 3 * E * H * 2
    big = lib.qmoe_moe_route_workspace_bytes(T, H, E, 8)
    assert big >= parts + 4 * T * E * 4
    small = lib.qmoe_moe_route_workspace_bytes(64, H, E, 8)
    assert small < parts
    # E not a multiple of 128: the CUDA-core router, partial logits only
    up256 = lambda n: (n + 255) // 256 * 256
    assert lib.qmoe_moe_route_workspace_bytes(T, H, 200, 8) in {up256(sp * T * 200 * 4) for sp in (1, 2, 4, 8)}


def test_threshold_roundtrip(lib):
    old = qb.get_gemm_threshold()
    qb.set_gemm_threshold(77)
    assert qb.get_gemm_threshold() == 77
    qb.set_gemm_threshold(-1)
    assert qb.get_gemm_threshold() == 2**31 - 1 or qb.get_gemm_threshold() > 0
    qb.set_gemm_threshold(old)
