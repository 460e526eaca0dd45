"""The allocation-free entry point against the regular one.

qmoe_moe_forward_noalloc serves callers that cannot allocate device memory
(plugin interfaces that pass only inputs and outputs, threads that must not
call cudaMalloc); it uses a fixed scratch array inside the library. This file
runs last so that a failure here leaves every other test already run.
"""

import ctypes

import numpy as np
import pytest
import torch

from quantized_moe_transformer_gb300 import binding as qb
from quantized_moe_transformer_gb300 import inputs
from tests.parity import TOL_GEMV, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def layer():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from quantized_moe_transformer_gb300 import build
    build.build()
    arr = inputs.moe_layer(3, 2048, 256, 512, shared=True)
    return qb.MoeLayer.from_arrays(arr, 8)


@pytest.mark.parametrize("T", [1, 16, 64])
def test_noalloc_matches_workspace_entry_point(layer, T):
    X = torch.from_numpy(inputs.hidden(40 + T, T, 2048)).cuda()
    ref = qb.moe_forward(layer, X, X)
    for _ in range(2):  # two calls in a row share the scratch
        got = qb.moe_forward_noalloc(layer, X, X)
        torch.cuda.synchronize()
        assert qb.query_status() == 0
        assert_close(got.cpu().numpy(), ref.cpu().numpy(), TOL_GEMV)
    X2 = torch.from_numpy(inputs.hidden(90 + T, T, 2048)).cuda()
    got2 = qb.moe_forward_noalloc(layer, X2)
    ref2 = qb.moe_forward(layer, X2)
    torch.cuda.synchronize()
    assert_close(got2.cpu().numpy(), ref2.cpu().numpy(), TOL_GEMV)


def test_noalloc_rejects_oversize(layer):
    T = 512
    assert layer.workspace_bytes(T) > (8 << 20)
    X = torch.zeros((T, 2048), device="cuda")
    out = torch.zeros_like(X)
    r = qb.lib().qmoe_moe_forward_noalloc(ctypes.byref(layer.desc), ctypes.c_void_p(X.data_ptr()), None,
                                          ctypes.c_void_p(out.data_ptr()), T, None)
    assert r == -10
    assert b"scratch" in qb.lib().qmoe_status_str(r)
    assert torch.count_nonzero(out).item() == 0


def _largest_fitting_rows(layer):
    T = 1
    while layer.workspace_bytes(T + 1) <= (8 << 20):
        T += 1
    return T


def test_noalloc_row_limit_boundary(layer):
    """The largest row count whose workspace fits the 8 MiB scratch runs and
    matches the workspace entry point; one row more is refused with
    QMOE_ERR_TOO_LARGE and leaves ``out`` untouched."""
    T = _largest_fitting_rows(layer)
    assert T == 86  # at this layer shape, as the header states
    X = torch.from_numpy(inputs.hidden(7, T, 2048)).cuda()
    ref = qb.moe_forward(layer, X)
    got = qb.moe_forward_noalloc(layer, X)
    torch.cuda.synchronize()
    assert qb.query_status() == 0
    assert_close(got.cpu().numpy(), ref.cpu().numpy(), TOL_GEMV)
    X1 = torch.from_numpy(inputs.hidden(8, T + 1, 2048)).cuda()
    out = torch.full_like(X1, 3.0)
    r = qb.lib().qmoe_moe_forward_noalloc(ctypes.byref(layer.desc), ctypes.c_void_p(X1.data_ptr()), None,
                                          ctypes.c_void_p(out.data_ptr()), T + 1, None)
    torch.cuda.synchronize()
    assert r == -10
    assert bool(torch.all(out == 3.0))
